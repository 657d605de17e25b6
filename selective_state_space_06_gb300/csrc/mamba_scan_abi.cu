// C ABI of libmambascan.so: argument validation, buffer sizing, launches, the host-buffer
// end-to-end call and error reporting. The contract is documented in include/mamba_scan.h.
#include <cuda_runtime.h>

#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>

#include "../../include/mamba_scan.h"
#include "scan_plan.h"

namespace mscan {

static constexpr size_t kAlignFloats = 64;  // 256-byte alignment of scratch regions

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool make_plan(int64_t batch, int64_t T, int64_t Di, int64_t N, Plan* pl) {
  if (batch < 1 || T < 1 || Di < 1 || N < 1) return false;
  if (N > kMaxState || batch > 65535) return false;
  if (T > INT32_MAX || Di > INT32_MAX) return false;
  const double btd = (double)batch * (double)T * (double)Di;
  const double btn = (double)batch * (double)T * (double)N;
  if (btd >= 2147483648.0 || btn >= 2147483648.0) return false;
  Plan p;
  p.batch = batch; p.T = T; p.Di = Di; p.N = N;
  p.NP = N <= 4 ? 4 : N <= 8 ? 8 : N <= 16 ? 16 : N <= 32 ? 32 : 64;
  p.nchunks = (int)((T + kChunk - 1) / kChunk);
  auto split = [&](PassPlan& q, int want) {
    if (want < 1) want = 1;
    if (want > p.nchunks) want = p.nchunks;
    q.seg_chunks = (p.nchunks + want - 1) / want;
    q.nseg = (p.nchunks + q.seg_chunks - 1) / q.seg_chunks;
  };
  auto pass = [&](int npt, int dpt) {
    PassPlan q;
    q.NPT = npt;
    q.G = p.NP / npt;
    q.DC = kWarps * (32 / q.G) * dpt;
    q.nblk = (int)((Di + q.DC - 1) / q.DC);
    return q;
  };
  auto by_target = [&](PassPlan q, int target) {
    const int64_t rows = (int64_t)batch * q.nblk;
    split(q, (int)std::min<int64_t>((target + rows - 1) / rows, p.nchunks));
    return q;
  };
  // Segments for a kernel with `slots` resident CTAs: the fewest chunk steps on the critical
  // path (whole waves times chunks per segment, plus about one chunk of start-up per CTA) plus
  // the pre-pass, which costs about a quarter of the main kernel per chunk and covers every
  // segment but the first.
  auto by_waves = [&](PassPlan q, int slots) {
    const int64_t rows = (int64_t)batch * q.nblk;
    double best = 1e300;
    int best_want = 1;
    for (int want = 1; want <= std::min(p.nchunks, 64); ++want) {
      const int sc = (p.nchunks + want - 1) / want;
      const int ns = (p.nchunks + sc - 1) / sc;
      const int64_t waves = (rows * ns + slots - 1) / slots;
      const double cost = (double)waves * (sc + 1) +
                          0.25 * (double)(ns - 1) / ns * (double)p.nchunks * rows / slots;
      if (cost < best - 1e-9) { best = cost; best_want = want; }
    }
    split(q, best_want);
    return q;
  };
  p.fwd = by_target(pass(states_per_thread_fwd(p.NP), kDPT), target_units_fwd(p.NP));
  if (p.NP >= kTmemMinNP)
    p.bwd = by_waves(pass(4, kTmemDPT), kTmemSlots);
  else
    p.bwd = by_target(pass(states_per_thread_bwd(p.NP), kDPT), target_units_bwd(p.NP));
  p.bwd.sub_chunks = p.bwd.seg_chunks;
  p.bwd.nsub = 1;
  if (p.NP >= kTmemMinNP && p.bwd.nseg > 1) {
    // pre-pass CTAs: batch x (the main kernel's channel blocks) x (segments 1 .. nseg-1) x nsub
    const int64_t base = (int64_t)batch * p.bwd.nblk * (p.bwd.nseg - 1);
    int64_t k = (kBwdAggTarget + base - 1) / base;
    k = std::max<int64_t>(1, std::min<int64_t>(k, p.bwd.seg_chunks));
    p.bwd.sub_chunks = (int)((p.bwd.seg_chunks + k - 1) / k);
    p.bwd.nsub = (p.bwd.seg_chunks + p.bwd.sub_chunks - 1) / p.bwd.sub_chunks;
  }
  const size_t bdn = (size_t)batch * (size_t)Di * (size_t)N;
  const size_t bd = (size_t)batch * (size_t)Di;
  size_t ck = round_up((size_t)(p.nchunks - 1) * bdn, kAlignFloats);
  if (p.fwd.nseg > 1) {
    p.off_fagg_h = ck; ck = round_up(ck + (size_t)p.fwd.nseg * bdn, kAlignFloats);
    p.off_fagg_sd = ck; ck = round_up(ck + (size_t)p.fwd.nseg * bd, kAlignFloats);
  }
  p.off_y = ck; ck = round_up(ck + (size_t)batch * (size_t)T * (size_t)Di, kAlignFloats);
  p.ckpt_elems = ck;
  const size_t part_bc = (size_t)p.bwd.nblk * (size_t)batch * (size_t)T * (size_t)N;
  size_t off = 0;
  p.off_partB = off; off = round_up(off + part_bc, kAlignFloats);
  p.off_partC = off; off = round_up(off + part_bc, kAlignFloats);
  p.off_partA = off; off = round_up(off + (size_t)p.bwd.nseg * bdn, kAlignFloats);
  p.off_partD = off; off = round_up(off + (size_t)p.bwd.nseg * bd, kAlignFloats);
  const size_t nslot = (size_t)p.bwd.nseg * p.bwd.nsub;
  p.off_bagg_L = off; off = round_up(off + nslot * bdn, kAlignFloats);
  p.off_bagg_sd = off; off = round_up(off + nslot * bd, kAlignFloats);
  p.scratch_elems = off;
  *pl = p;
  return true;
}

}  // namespace mscan

using mscan::Plan;
using mscan::round_up;

namespace {

thread_local int g_last_launches = 0;
thread_local cudaError_t g_last_cuda = cudaSuccess;

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

struct Range {
  uintptr_t lo, hi;
};

bool overlaps(const Range& a, const Range& b) { return a.lo < b.hi && b.lo < a.hi; }

int set_cuda_error(cudaError_t e) {
  g_last_cuda = e;
  return MAMBA_ERR_CUDA;
}

// Common size/pointer checks of the device entry points.
int check_dims(int64_t batch, int64_t T, int64_t Di, int64_t N, Plan* plan) {
  if (N > mscan::kMaxState && batch >= 1 && T >= 1 && Di >= 1) return MAMBA_ERR_UNSUPPORTED;
  if (!mscan::make_plan(batch, T, Di, N, plan)) return MAMBA_ERR_INVALID_ARG;
  return MAMBA_OK;
}

}  // namespace

extern "C" {

size_t mamba_scan_ckpt_bytes(int64_t batch, int64_t T, int64_t d_inner, int64_t d_state) {
  Plan p;
  if (!mscan::make_plan(batch, T, d_inner, d_state, &p)) return 0;
  return p.ckpt_elems * sizeof(float);
}

size_t mamba_scan_scratch_bytes(int64_t batch, int64_t T, int64_t d_inner, int64_t d_state) {
  Plan p;
  if (!mscan::make_plan(batch, T, d_inner, d_state, &p)) return 0;
  return p.scratch_elems * sizeof(float);
}

int mamba_scan_fwd(const float* delta, const float* u, const float* B, const float* C,
                   const float* gate, const float* A_log, const float* D, float* out, float* y,
                   void* ckpt, size_t ckpt_bytes, int64_t batch, int64_t T, int64_t d_inner,
                   int64_t d_state, void* stream) {
  Plan plan;
  int rc = check_dims(batch, T, d_inner, d_state, &plan);
  if (rc != MAMBA_OK) return rc;
  const size_t need_ck = plan.ckpt_elems * sizeof(float);
  if (!delta || !u || !B || !C || !gate || !A_log || !D || !out) return MAMBA_ERR_INVALID_ARG;
  if (need_ck > 0 && !ckpt) return MAMBA_ERR_INVALID_ARG;
  const void* ptrs[] = {delta, u, B, C, gate, A_log, D, out, y, ckpt};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return MAMBA_ERR_MISALIGNED;
  if (ckpt_bytes < need_ck) return MAMBA_ERR_WORKSPACE;
  const size_t btd = (size_t)batch * T * d_inner * sizeof(float);
  {
    Range ro = {(uintptr_t)out, (uintptr_t)out + btd};
    if (y && overlaps(ro, Range{(uintptr_t)y, (uintptr_t)y + btd})) return MAMBA_ERR_INVALID_ARG;
    if (need_ck && overlaps(ro, Range{(uintptr_t)ckpt, (uintptr_t)ckpt + need_ck}))
      return MAMBA_ERR_INVALID_ARG;
  }
  mscan::FwdParams p;
  p.delta = delta; p.u = u; p.B = B; p.C = C; p.gate = gate; p.A_log = A_log; p.D = D;
  p.out = out; p.y = y; p.ckpt = (float*)ckpt;
  p.agg_h = plan.fwd.nseg > 1 ? (float*)ckpt + plan.off_fagg_h : nullptr;
  p.agg_sd = plan.fwd.nseg > 1 ? (float*)ckpt + plan.off_fagg_sd : nullptr;
  p.y_ck = (float*)ckpt + plan.off_y;
  p.batch = (int)batch; p.T = (int)T; p.Di = (int)d_inner; p.N = (int)d_state;
  p.nchunks = plan.nchunks; p.nblk = plan.fwd.nblk;
  p.seg_chunks = plan.fwd.seg_chunks; p.nseg = plan.fwd.nseg;
  const int n = mscan::launch_fwd(plan, p, (cudaStream_t)stream);
  if (n < 0) return set_cuda_error(cudaGetLastError());
  g_last_launches = n;
  return MAMBA_OK;
}

int mamba_scan_bwd(const float* delta, const float* u, const float* B, const float* C,
                   const float* gate, const float* A_log, const float* D, const float* dy,
                   const void* ckpt, size_t ckpt_bytes, void* scratch, size_t scratch_bytes,
                   float* d_delta, float* d_u, float* d_B, float* d_C, float* d_A_log,
                   float* d_D, float* d_gate, int64_t batch, int64_t T, int64_t d_inner,
                   int64_t d_state, void* stream) {
  Plan plan;
  int rc = check_dims(batch, T, d_inner, d_state, &plan);
  if (rc != MAMBA_OK) return rc;
  const size_t need_ck = plan.ckpt_elems * sizeof(float);
  const size_t need_sc = plan.scratch_elems * sizeof(float);
  if (!delta || !u || !B || !C || !gate || !A_log || !D || !dy || !scratch || !d_delta ||
      !d_u || !d_B || !d_C || !d_A_log || !d_D || !d_gate)
    return MAMBA_ERR_INVALID_ARG;
  if (need_ck > 0 && !ckpt) return MAMBA_ERR_INVALID_ARG;
  const void* ptrs[] = {delta, u, B, C, gate, A_log, D, dy, ckpt, scratch,
                        d_delta, d_u, d_B, d_C, d_A_log, d_D, d_gate};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return MAMBA_ERR_MISALIGNED;
  if (ckpt_bytes < need_ck || scratch_bytes < need_sc) return MAMBA_ERR_WORKSPACE;
  {
    const size_t btd = (size_t)batch * T * d_inner * sizeof(float);
    const size_t btn = (size_t)batch * T * d_state * sizeof(float);
    const Range outs[] = {
        {(uintptr_t)d_delta, (uintptr_t)d_delta + btd},
        {(uintptr_t)d_u, (uintptr_t)d_u + btd},
        {(uintptr_t)d_gate, (uintptr_t)d_gate + btd},
        {(uintptr_t)d_B, (uintptr_t)d_B + btn},
        {(uintptr_t)d_C, (uintptr_t)d_C + btn},
        {(uintptr_t)d_A_log, (uintptr_t)d_A_log + (size_t)d_inner * d_state * sizeof(float)},
        {(uintptr_t)d_D, (uintptr_t)d_D + (size_t)d_inner * sizeof(float)},
        {(uintptr_t)scratch, (uintptr_t)scratch + need_sc},
        {(uintptr_t)ckpt, (uintptr_t)ckpt + need_ck},
    };
    const int nout = need_ck ? 9 : 8;
    for (int i = 0; i < nout; ++i)
      for (int j = i + 1; j < nout; ++j)
        if (overlaps(outs[i], outs[j])) return MAMBA_ERR_INVALID_ARG;
  }
  float* sc = (float*)scratch;
  mscan::BwdParams p;
  p.delta = delta; p.u = u; p.B = B; p.C = C; p.gate = gate; p.A_log = A_log; p.D = D;
  p.dy = dy; p.ckpt = (const float*)ckpt; p.y_ck = (const float*)ckpt + plan.off_y;
  p.d_delta = d_delta; p.d_u = d_u; p.d_gate = d_gate;
  p.partB = sc + plan.off_partB; p.partC = sc + plan.off_partC;
  p.partA = sc + plan.off_partA; p.partD = sc + plan.off_partD;
  p.agg_L = sc + plan.off_bagg_L; p.agg_sd = sc + plan.off_bagg_sd;
  p.d_B = d_B; p.d_C = d_C; p.d_A_log = d_A_log; p.d_D = d_D;
  p.batch = (int)batch; p.T = (int)T; p.Di = (int)d_inner; p.N = (int)d_state;
  p.nchunks = plan.nchunks; p.nblk = plan.bwd.nblk;
  p.seg_chunks = plan.bwd.seg_chunks; p.nseg = plan.bwd.nseg;
  p.sub_chunks = plan.bwd.sub_chunks; p.nsub = plan.bwd.nsub;
  const int n = mscan::launch_bwd(plan, p, (cudaStream_t)stream);
  if (n < 0) return set_cuda_error(cudaGetLastError());
  g_last_launches = n;
  return MAMBA_OK;
}

size_t mamba_scan_host_workspace_bytes(int64_t batch, int64_t T, int64_t d_inner,
                                       int64_t d_state) {
  Plan p;
  if (!mscan::make_plan(batch, T, d_inner, d_state, &p)) return 0;
  const size_t a = 256;
  const size_t btd = round_up((size_t)batch * T * d_inner * sizeof(float), a);
  const size_t btn = round_up((size_t)batch * T * d_state * sizeof(float), a);
  const size_t dn = round_up((size_t)d_inner * d_state * sizeof(float), a);
  const size_t dd = round_up((size_t)d_inner * sizeof(float), a);
  // inputs: delta u gate dy (4 btd), B C (2 btn), A_log, D
  // outputs: out d_delta d_u d_gate (4 btd), d_B d_C (2 btn), d_A_log, d_D
  return 8 * btd + 4 * btn + 2 * dn + 2 * dd + round_up(p.ckpt_elems * sizeof(float), a) +
         round_up(p.scratch_elems * sizeof(float), a);
}

int mamba_scan_fwd_bwd_host(const float* delta, const float* u, const float* B, const float* C,
                            const float* gate, const float* A_log, const float* D,
                            const float* dy, float* out, float* d_delta, float* d_u, float* d_B,
                            float* d_C, float* d_A_log, float* d_D, float* d_gate,
                            void* workspace, size_t workspace_bytes, int64_t batch, int64_t T,
                            int64_t d_inner, int64_t d_state, void* stream) {
  Plan plan;
  int rc = check_dims(batch, T, d_inner, d_state, &plan);
  if (rc != MAMBA_OK) return rc;
  if (!delta || !u || !B || !C || !gate || !A_log || !D || !dy || !out || !d_delta || !d_u ||
      !d_B || !d_C || !d_A_log || !d_D || !d_gate || !workspace)
    return MAMBA_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return MAMBA_ERR_MISALIGNED;
  if (workspace_bytes < mamba_scan_host_workspace_bytes(batch, T, d_inner, d_state))
    return MAMBA_ERR_WORKSPACE;
  const size_t a = 256;
  const size_t btd = (size_t)batch * T * d_inner * sizeof(float);
  const size_t btn = (size_t)batch * T * d_state * sizeof(float);
  const size_t dn = (size_t)d_inner * d_state * sizeof(float);
  const size_t dd = (size_t)d_inner * sizeof(float);
  char* w = (char*)workspace;
  auto take = [&](size_t bytes) {
    char* q = w;
    w += round_up(bytes, a);
    return (float*)q;
  };
  float *w_delta = take(btd), *w_u = take(btd), *w_gate = take(btd), *w_dy = take(btd);
  float *w_B = take(btn), *w_C = take(btn), *w_A = take(dn), *w_D = take(dd);
  float *w_out = take(btd), *w_dd = take(btd), *w_du = take(btd), *w_dg = take(btd);
  float *w_dB = take(btn), *w_dC = take(btn), *w_dA = take(dn), *w_dD = take(dd);
  const size_t ck_bytes = plan.ckpt_elems * sizeof(float);
  const size_t sc_bytes = plan.scratch_elems * sizeof(float);
  float* w_ck = take(ck_bytes);
  float* w_sc = take(sc_bytes);
  cudaStream_t s = (cudaStream_t)stream;
  struct Cp { void* dst; const void* src; size_t n; };
  const Cp h2d[] = {{w_delta, delta, btd}, {w_u, u, btd},   {w_gate, gate, btd},
                    {w_dy, dy, btd},       {w_B, B, btn},   {w_C, C, btn},
                    {w_A, A_log, dn},      {w_D, D, dd}};
  for (const Cp& c : h2d) {
    cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  rc = mamba_scan_fwd(w_delta, w_u, w_B, w_C, w_gate, w_A, w_D, w_out, nullptr,
                      ck_bytes ? w_ck : nullptr, ck_bytes, batch, T, d_inner, d_state, stream);
  if (rc != MAMBA_OK) return rc;
  const int nf = g_last_launches;
  rc = mamba_scan_bwd(w_delta, w_u, w_B, w_C, w_gate, w_A, w_D, w_dy, ck_bytes ? w_ck : nullptr,
                      ck_bytes, w_sc, sc_bytes, w_dd, w_du, w_dB, w_dC, w_dA, w_dD, w_dg, batch,
                      T, d_inner, d_state, stream);
  if (rc != MAMBA_OK) return rc;
  g_last_launches += nf;
  const Cp d2h[] = {{out, w_out, btd},   {d_delta, w_dd, btd}, {d_u, w_du, btd},
                    {d_gate, w_dg, btd}, {d_B, w_dB, btn},     {d_C, w_dC, btn},
                    {d_A_log, w_dA, dn}, {d_D, w_dD, dd}};
  for (const Cp& c : d2h) {
    cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_cuda_error(e);
  if (mscan::bwd_take_fault()) return MAMBA_ERR_TIMEOUT;
  return MAMBA_OK;
}

int mamba_scan_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return set_cuda_error(e);
  if (mscan::bwd_take_fault()) return MAMBA_ERR_TIMEOUT;
  return MAMBA_OK;
}

const char* mamba_scan_strerror(int code) {
  switch (code) {
    case MAMBA_OK: return "ok";
    case MAMBA_ERR_INVALID_ARG:
      return "invalid argument (null pointer, size out of range, or overlapping outputs)";
    case MAMBA_ERR_MISALIGNED: return "a pointer is not 16-byte aligned";
    case MAMBA_ERR_WORKSPACE: return "checkpoint, scratch or workspace buffer too small";
    case MAMBA_ERR_CUDA: return cudaGetErrorString(g_last_cuda);
    case MAMBA_ERR_UNSUPPORTED: return "d_state outside 1..64 is not supported";
    case MAMBA_ERR_NOALLOC_LIMIT:
      return "mamba_scan_bwd_noalloc: these sizes need more scratch than the static 64 MiB array";
    case MAMBA_ERR_TIMEOUT:
      return "a kernel gave up waiting for its asynchronous copies; recent outputs are invalid";
    default: return "unknown error code";
  }
}

int mamba_scan_last_launch_count(void) { return g_last_launches; }

}  // extern "C"
