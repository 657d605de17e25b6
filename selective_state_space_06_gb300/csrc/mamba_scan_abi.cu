// C ABI of libmambascan.so: argument validation, buffer sizing, launches, the host-buffer
// end-to-end call and error reporting. The contract is documented in include/mamba_scan.h.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>   // header-only; ranges cost a pointer check when no tool listens

#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "../../include/mamba_scan.h"
#include "scan_plan.h"

using mscan::Plan;
using mscan::round_up;

namespace mscan {
// An NVTX range around one entry point call (visible in Nsight Systems / ncu range filters).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace mscan

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

// the bounds-checked build's fault words of every kernel file, read and cleared (0 in the
// default build, without any CUDA call)
unsigned int take_oob() {
  return mscan::fwd_take_oob() | mscan::bwd_take_oob() | mscan::tmem_take_oob() |
         mscan::conv_take_oob();
}

}  // namespace

namespace mscan {
int record_cuda_error(cudaError_t e) { return set_cuda_error(e); }
}  // namespace mscan

namespace {

// Common size/pointer checks of the device entry points.
int check_dims(int64_t batch, int64_t T, int64_t Di, int64_t N, Plan* plan) {
  if (N > mscan::kMaxState && batch >= 1 && T >= 1 && Di >= 1) return MAMBA_ERR_UNSUPPORTED;
  if (!mscan::make_plan(batch, T, Di, N, plan)) return MAMBA_ERR_INVALID_ARG;
  return MAMBA_OK;
}

// Device workspace of mamba_scan_fwd_bwd_host: the whole batch's inputs and outputs, then one
// set of checkpoint + scratch buffers per slice, then the slices' d_A_log / d_D sums.
// At most kHostSlices slices (streams, workspace regions); a batch is cut into at most
// kBatchSlices slices of whole rows.
constexpr int kHostSlices = 8;
constexpr int kBatchSlices = 4;

// A batch smaller than the slice count is cut into blocks of channels instead (each slice is
// then the whole batch over dcs consecutive channels, a scan of its own); the smallest block
// worth a slice of its own:
constexpr int64_t kMinSliceChannels = 64;
// Channel slices: at most kChanSlices, the first and the last half as wide as the others. The
// pipeline's head (the first slice's copies in) and tail (the last slice's kernels and copies
// out) then take half as long, while the middle slices keep rows wide enough for 2-D copies at
// the link's full rate (rows of 1280 bytes copy 15-20 % slower than rows of 2048 bytes and up).
constexpr int kChanSlices = 6;

struct HostLayout {
  int64_t rows = 0;            // batch rows per slice
  int nslices = 0;
  size_t off_in[8], off_out[8], off_ck[kHostSlices], off_sc[kHostSlices], off_part = 0;
  size_t ck_bytes = 0, sc_bytes = 0, total = 0;
  size_t dn_pad = 0, dd_pad = 0;   // floats
  // channel slices: each slice's compact inputs and outputs [batch][T][dcs], its A_log / D
  // rows and d_A_log / d_D rows (one region per slice), the shared B and C, and the slices'
  // d_B | d_C partials with their fixed-order sum
  bool by_channels = false;
  int64_t dcs = 0;                     // the widest slice's channels
  int64_t sd0[kHostSlices] = {}, sdw[kHostSlices] = {};   // each slice's first channel, width
  size_t off_slice[kHostSlices] = {};
  size_t sl_in[4] = {}, sl_A = 0, sl_D = 0, sl_out[4] = {}, sl_dA = 0, sl_dD = 0;   // in a slice
  size_t off_bc = 0, off_bcpart = 0, off_bcsum = 0;
};

static bool host_layout_channels(int64_t batch, int64_t T, int64_t Di, int64_t N,
                                 HostLayout* L) {
  HostLayout h;
  h.by_channels = true;
  // n slices of widths u, 2u, ..., 2u and the rest (about u), u a multiple of 4 and at least
  // kMinSliceChannels (the caller takes d_inner >= 2 * kMinSliceChannels, a multiple of 4)
  const int n = (int)std::max<int64_t>(
      2, std::min<int64_t>(kChanSlices, Di / (2 * kMinSliceChannels) + 1));
  const int64_t unit = Di / (2 * (n - 1)) / 4 * 4;
  int64_t d0 = 0;
  for (int k = 0; k < n; ++k) {
    const int64_t w = k == n - 1 ? Di - d0 : (k == 0 ? unit : 2 * unit);
    h.sd0[k] = d0;
    h.sdw[k] = w;
    h.dcs = std::max(h.dcs, w);
    d0 += w;
  }
  h.nslices = n;
  h.rows = batch;
  // checkpoint and scratch buffers sized for every slice's plan (a narrower slice may cut its
  // time axis into more segments)
  for (int k = 0; k < n; ++k) {
    Plan slice;
    if (!mscan::make_plan(batch, T, h.sdw[k], N, &slice)) return false;
    h.ck_bytes = std::max(h.ck_bytes, slice.ckpt_elems * sizeof(float));
    h.sc_bytes = std::max(h.sc_bytes, slice.scratch_elems * sizeof(float));
  }
  const size_t a = 256;
  const size_t btd_s = (size_t)batch * T * h.dcs * 4, btn = (size_t)batch * T * N * 4;
  size_t off = 0;   // inside one slice region
  for (int i = 0; i < 4; ++i) { h.sl_in[i] = off; off = round_up(off + btd_s, a); }
  h.sl_A = off; off = round_up(off + (size_t)h.dcs * N * 4, a);
  h.sl_D = off; off = round_up(off + (size_t)h.dcs * 4, a);
  for (int i = 0; i < 4; ++i) { h.sl_out[i] = off; off = round_up(off + btd_s, a); }
  h.sl_dA = off; off = round_up(off + (size_t)h.dcs * N * 4, a);
  h.sl_dD = off; off = round_up(off + (size_t)h.dcs * 4, a);
  const size_t slice_bytes = off;
  off = 0;
  for (int k = 0; k < h.nslices; ++k) {
    h.off_slice[k] = off; off = round_up(off + slice_bytes, a);
    h.off_ck[k] = off; off = round_up(off + h.ck_bytes, a);
    h.off_sc[k] = off; off = round_up(off + h.sc_bytes, a);
  }
  h.off_bc = off; off = round_up(off + 2 * btn, a);
  h.off_bcpart = off; off = round_up(off + (size_t)h.nslices * 2 * btn, a);
  h.off_bcsum = off; off = round_up(off + 2 * btn, a);
  h.total = off;
  *L = h;
  return true;
}

bool host_layout(int64_t batch, int64_t T, int64_t Di, int64_t N, HostLayout* L) {
  Plan whole;
  if (!mscan::make_plan(batch, T, Di, N, &whole)) return false;
  if (batch < kBatchSlices && Di % 4 == 0 && Di >= 2 * kMinSliceChannels)
    return host_layout_channels(batch, T, Di, N, L);
  HostLayout h;
  // slices start on 16-byte boundaries only when a batch row is a multiple of 4 floats
  const bool sliceable = (T * Di) % 4 == 0 && (T * N) % 4 == 0;
  h.nslices = sliceable ? (int)std::min<int64_t>(batch, kBatchSlices) : 1;
  h.rows = (batch + h.nslices - 1) / h.nslices;
  h.nslices = (int)((batch + h.rows - 1) / h.rows);
  Plan slice;
  if (!mscan::make_plan(h.rows, T, Di, N, &slice)) return false;
  // a shorter last slice needs no more checkpoint or scratch than a full one
  h.ck_bytes = slice.ckpt_elems * sizeof(float);
  h.sc_bytes = slice.scratch_elems * sizeof(float);
  const size_t a = 256;
  const size_t btd = (size_t)batch * T * Di * 4, btn = (size_t)batch * T * N * 4;
  // d_A_log | d_D of one slice, each padded to 16 bytes
  h.dn_pad = round_up((size_t)Di * N, 4);
  h.dd_pad = round_up((size_t)Di, 4);
  const size_t dn = (size_t)Di * N * 4, dd = (size_t)Di * 4;
  const size_t part = (h.dn_pad + h.dd_pad) * 4;
  const size_t in_sz[8] = {btd, btd, btd, btd, btn, btn, dn, dd};    // delta u gate dy B C A D
  const size_t out_sz[8] = {btd, btd, btd, btd, btn, btn, part, 0};   // out dd du dg dB dC dA|dD
  size_t off = 0;
  for (int i = 0; i < 8; ++i) { h.off_in[i] = off; off = round_up(off + in_sz[i], a); }
  for (int i = 0; i < 8; ++i) { h.off_out[i] = off; off = round_up(off + out_sz[i], a); }
  for (int i = 0; i < h.nslices; ++i) {
    h.off_ck[i] = off; off = round_up(off + h.ck_bytes, a);
    h.off_sc[i] = off; off = round_up(off + h.sc_bytes, a);
  }
  h.off_part = off; off = round_up(off + (size_t)h.nslices * part, a);
  h.total = off;
  *L = h;
  return true;
}

// The library's extra streams (one per slice after the first) and one event per slice on the
// current device, created once per device.
struct AuxStreams {
  cudaStream_t s[kHostSlices] = {};
  cudaEvent_t ev[kHostSlices + 1] = {};      // slice done; [kHostSlices]: A_log, D copied
  cudaEvent_t ev_in[kHostSlices] = {};       // slice's host->device copies done
  cudaEvent_t ev_out[kHostSlices] = {};      // slice's device->host copies done
  // channel slices: the device->host copies go on a stream of their own, in slice order
  cudaStream_t d2h = nullptr;
  cudaEvent_t ev_fwd[kHostSlices] = {};      // slice's forward done (out is final)
  cudaEvent_t ev_bwd[kHostSlices] = {};      // slice's backward done
  cudaEvent_t ev_end = nullptr;              // the last device->host copy done
  // Held by a call from its first enqueue to its return. Calls from several host threads share
  // these streams and events, and an event recorded by one call must not be re-recorded by
  // another between that record and the waits on it (on the caller's own stream, such a
  // re-record would point the waits at the other call's work). Held through the final
  // synchronisation too, so that the fault words read after it belong to this call.
  std::mutex* enqueue = nullptr;
};
bool aux_streams(AuxStreams* out) {
  static std::mutex mu;
  static std::mutex enqueue_mu[64];
  static AuxStreams aux[64];
  static bool ready[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  AuxStreams& x = aux[dev];
  x.enqueue = &enqueue_mu[dev];
  if (!ready[dev]) {
    for (int i = 1; i < kHostSlices; ++i)
      if (cudaStreamCreateWithFlags(&x.s[i], cudaStreamNonBlocking) != cudaSuccess) return false;
    for (int i = 0; i <= kHostSlices; ++i)
      if (cudaEventCreateWithFlags(&x.ev[i], cudaEventDisableTiming) != cudaSuccess) return false;
    for (int i = 0; i < kHostSlices; ++i)
      if (cudaEventCreateWithFlags(&x.ev_in[i], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&x.ev_out[i], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&x.ev_fwd[i], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&x.ev_bwd[i], cudaEventDisableTiming) != cudaSuccess)
        return false;
    if (cudaStreamCreateWithFlags(&x.d2h, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&x.ev_end, cudaEventDisableTiming) != cudaSuccess)
      return false;
    ready[dev] = true;
  }
  *out = x;
  return true;
}

}  // namespace

namespace mscan {
// out[i] = sum over slices k (in order) of part[k][i]
__global__ void sum_slices(const float* part, int nslices, size_t n, float* out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    float acc = 0.f;
    for (int k = 0; k < nslices; ++k) acc += part[(size_t)k * n + i];
    out[i] = acc;
  }
}
}  // namespace mscan

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

static int scan_fwd_impl(const float* delta, const float* u, const float* B, const float* C,
                         const float* gate, const float* A_log, const float* D, float* out,
                         float* y, void* ckpt, size_t ckpt_bytes, int64_t batch, int64_t T,
                         int64_t d_inner, int64_t d_state, void* stream, int softplus,
                         int states_only = 0, int io_bf16 = 0, int test_timeout = 0) {
  Plan plan;
  int rc = check_dims(batch, T, d_inner, d_state, &plan);
  if (rc != MAMBA_OK) return rc;
  const size_t need_ck = plan.ckpt_elems * sizeof(float);
  if (!delta || !u || !B || !C || !gate || !A_log || !D || (!out && !states_only))
    return MAMBA_ERR_INVALID_ARG;
  if (need_ck > 0 && !ckpt) return MAMBA_ERR_INVALID_ARG;
  const void* ptrs[] = {delta, u, B, C, gate, A_log, D, out, y, ckpt};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return MAMBA_ERR_MISALIGNED;
  if (ckpt_bytes < need_ck) return MAMBA_ERR_WORKSPACE;
  const size_t btd = (size_t)batch * T * d_inner * (io_bf16 ? 2 : sizeof(float));
  if (out) {
    Range ro = {(uintptr_t)out, (uintptr_t)out + btd};
    if (y && overlaps(ro, Range{(uintptr_t)y, (uintptr_t)y + btd})) return MAMBA_ERR_INVALID_ARG;
    if (need_ck && overlaps(ro, Range{(uintptr_t)ckpt, (uintptr_t)ckpt + need_ck}))
      return MAMBA_ERR_INVALID_ARG;
  }
  mscan::FwdParams p = {};
  p.delta = delta; p.u = u; p.B = B; p.C = C; p.gate = gate; p.A_log = A_log; p.D = D;
  p.out = out; p.y = y; p.ckpt = (float*)ckpt;
  p.agg_h = plan.fwd.nseg > 1 ? (float*)ckpt + plan.off_fagg_h : nullptr;
  p.agg_sd = plan.fwd.nseg > 1 ? (float*)ckpt + plan.off_fagg_sd : nullptr;
  p.y_ck = (float*)ckpt + plan.off_y;
  p.batch = (int)batch; p.T = (int)T; p.Di = (int)d_inner; p.N = (int)d_state;
  p.nchunks = plan.nchunks; p.nblk = plan.fwd.nblk;
  p.seg_chunks = plan.fwd.seg_chunks; p.nseg = plan.fwd.nseg;
  p.agg_k = 1;
  p.softplus = softplus;
  p.states_only = states_only;
  p.io_bf16 = io_bf16;
  p.wait_limit_ns = 1000000000ull;   // one second per copy wait
  if (test_timeout) {
    // the failure-path test: the forward with tensor copies leaves the copies of each CTA's
    // last chunk unissued and gives up waiting for them after 1 ms
    p.test_skip_last_copy = 1;
    p.wait_limit_ns = 1000000ull;
  }
  const int n = mscan::launch_fwd(plan, p, (cudaStream_t)stream);
  if (n < 0) return set_cuda_error(cudaGetLastError());
  g_last_launches = n;
  return MAMBA_OK;
}

int mamba_scan_fwd(const float* delta, const float* u, const float* B, const float* C,
                   const float* gate, const float* A_log, const float* D, float* out, float* y,
                   void* ckpt, size_t ckpt_bytes, int64_t batch, int64_t T, int64_t d_inner,
                   int64_t d_state, void* stream) {
  mscan::NvtxRange nvtx_range("mamba_scan_fwd");
  return scan_fwd_impl(delta, u, B, C, gate, A_log, D, out, y, ckpt, ckpt_bytes, batch, T,
                       d_inner, d_state, stream, 0);
}

int mamba_scan_fwd_test_timeout(const float* delta, const float* u, const float* B,
                                const float* C, const float* gate, const float* A_log,
                                const float* D, float* out, float* y, void* ckpt,
                                size_t ckpt_bytes, int64_t batch, int64_t T, int64_t d_inner,
                                int64_t d_state, void* stream) {
  mscan::NvtxRange nvtx_range("mamba_scan_fwd_test_timeout");
  Plan plan;
  const int rc = check_dims(batch, T, d_inner, d_state, &plan);
  if (rc != MAMBA_OK) return rc;
  // only the forward with tensor-copy staging (d_state 33..64, d_inner and d_state multiples
  // of 4) waits on copies it issues itself
  if (plan.NP != mscan::kMaxState || d_inner % 4 != 0 || d_state % 4 != 0 || plan.nchunks < 2)
    return MAMBA_ERR_UNSUPPORTED;
  return scan_fwd_impl(delta, u, B, C, gate, A_log, D, out, y, ckpt, ckpt_bytes, batch, T,
                       d_inner, d_state, stream, 0, 0, 0, 1);
}

int mamba_scan_fwd_softplus(const float* delta_raw, const float* u, const float* B,
                            const float* C, const float* gate, const float* A_log,
                            const float* D, float* out, float* y, void* ckpt,
                            size_t ckpt_bytes, int64_t batch, int64_t T, int64_t d_inner,
                            int64_t d_state, void* stream) {
  mscan::NvtxRange nvtx_range("mamba_scan_fwd_softplus");
  return scan_fwd_impl(delta_raw, u, B, C, gate, A_log, D, out, y, ckpt, ckpt_bytes, batch, T,
                       d_inner, d_state, stream, 1);
}

static int scan_bwd_impl(const float* delta, const float* u, const float* B, const float* C,
                         const float* gate, const float* A_log, const float* D, const float* dy,
                         const void* ckpt, size_t ckpt_bytes, void* scratch,
                         size_t scratch_bytes, float* d_delta, float* d_u, float* d_B,
                         float* d_C, float* d_A_log, float* d_D, float* d_gate, int64_t batch,
                         int64_t T, int64_t d_inner, int64_t d_state, void* stream,
                         int softplus, float* out = nullptr, bool fuse_out = false,
                         bool check_only = false, int io_bf16 = 0, int phase = 0,
                         void* pre_stream = nullptr, int test_timeout = 0) {
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
                        d_delta, d_u, d_B, d_C, d_A_log, d_D, d_gate, out};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return MAMBA_ERR_MISALIGNED;
  if (ckpt_bytes < need_ck || scratch_bytes < need_sc) return MAMBA_ERR_WORKSPACE;
  {
    const size_t es = io_bf16 ? 2 : sizeof(float);   // element size of the I/O tensors
    const size_t btd = (size_t)batch * T * d_inner * es;
    const size_t btn = (size_t)batch * T * d_state * es;
    const Range outs[] = {
        {(uintptr_t)d_delta, (uintptr_t)d_delta + btd},
        {(uintptr_t)d_u, (uintptr_t)d_u + btd},
        {(uintptr_t)d_gate, (uintptr_t)d_gate + btd},
        {(uintptr_t)d_B, (uintptr_t)d_B + btn},
        {(uintptr_t)d_C, (uintptr_t)d_C + btn},
        {(uintptr_t)d_A_log, (uintptr_t)d_A_log + (size_t)d_inner * d_state * sizeof(float)},
        {(uintptr_t)d_D, (uintptr_t)d_D + (size_t)d_inner * sizeof(float)},
        {(uintptr_t)scratch, (uintptr_t)scratch + need_sc},
        {(uintptr_t)out, (uintptr_t)out + (out ? btd : 0)},
        {(uintptr_t)ckpt, (uintptr_t)ckpt + need_ck},
    };
    const int nout = need_ck ? 10 : 9;
    for (int i = 0; i < nout; ++i)
      for (int j = i + 1; j < nout; ++j)
        if (overlaps(outs[i], outs[j])) return MAMBA_ERR_INVALID_ARG;
  }
  if (check_only) return MAMBA_OK;
  float* sc = (float*)scratch;
  mscan::BwdParams p = {};
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
  p.softplus = softplus;
  p.out = fuse_out ? out : nullptr;
  if (fuse_out) p.y_ck = nullptr;   // y is recomputed from the states
  p.io_bf16 = io_bf16;
  p.wait_limit_ns = 1000000000ull;   // one second per copy wait
  if (test_timeout) {
    // the failure-path test: the tensor-memory backward leaves the copies of each CTA's last
    // chunk unissued and gives up waiting for them after 1 ms
    p.test_skip_last_copy = 1;
    p.wait_limit_ns = 1000000ull;
  }
  // phase 0: everything on `stream`; 1: the segment pre-pass and the composition of the
  // carries, on `pre_stream`; 2: the backward and the reduction, on `stream` (d_state 9..64)
  const int n = phase == 1   ? mscan::launch_bwd_carries(plan, p, (cudaStream_t)pre_stream)
                : phase == 2 ? mscan::launch_bwd_after_carries(plan, p, (cudaStream_t)stream)
                             : mscan::launch_bwd(plan, p, (cudaStream_t)stream);
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
  mscan::NvtxRange nvtx_range("mamba_scan_bwd");
  return scan_bwd_impl(delta, u, B, C, gate, A_log, D, dy, ckpt, ckpt_bytes, scratch,
                       scratch_bytes, d_delta, d_u, d_B, d_C, d_A_log, d_D, d_gate, batch, T,
                       d_inner, d_state, stream, 0);
}

int mamba_scan_bwd_softplus(const float* delta_raw, const float* u, const float* B,
                            const float* C, const float* gate, const float* A_log,
                            const float* D, const float* dy, const void* ckpt,
                            size_t ckpt_bytes, void* scratch, size_t scratch_bytes,
                            float* d_delta_raw, float* d_u, float* d_B, float* d_C,
                            float* d_A_log, float* d_D, float* d_gate, int64_t batch, int64_t T,
                            int64_t d_inner, int64_t d_state, void* stream) {
  mscan::NvtxRange nvtx_range("mamba_scan_bwd_softplus");
  return scan_bwd_impl(delta_raw, u, B, C, gate, A_log, D, dy, ckpt, ckpt_bytes, scratch,
                       scratch_bytes, d_delta_raw, d_u, d_B, d_C, d_A_log, d_D, d_gate, batch,
                       T, d_inner, d_state, stream, 1);
}

int mamba_scan_bwd_test_timeout(const float* delta, const float* u, const float* B,
                                const float* C, const float* gate, const float* A_log,
                                const float* D, const float* dy, const void* ckpt,
                                size_t ckpt_bytes, void* scratch, size_t scratch_bytes,
                                float* d_delta, float* d_u, float* d_B, float* d_C,
                                float* d_A_log, float* d_D, float* d_gate, int64_t batch,
                                int64_t T, int64_t d_inner, int64_t d_state, void* stream) {
  mscan::NvtxRange nvtx_range("mamba_scan_bwd_test_timeout");
  Plan plan;
  const int rc = check_dims(batch, T, d_inner, d_state, &plan);
  if (rc != MAMBA_OK) return rc;
  // only the tensor-memory backward with tensor-copy staging waits on copies it issues itself
  if (plan.NP < mscan::kTmemMinNP || d_inner % 4 != 0 || d_state % 4 != 0 || plan.nchunks < 2)
    return MAMBA_ERR_UNSUPPORTED;
  return scan_bwd_impl(delta, u, B, C, gate, A_log, D, dy, ckpt, ckpt_bytes, scratch,
                       scratch_bytes, d_delta, d_u, d_B, d_C, d_A_log, d_D, d_gate, batch, T,
                       d_inner, d_state, stream, 0, nullptr, false, false, 0, 0, nullptr, 1);
}

// The fused call's side stream and its two events, one set per (host thread, device), created
// on first use and kept for the thread's lifetime.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
static bool side_stream(SideStream* out) {
  thread_local SideStream per_dev[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  SideStream& x = per_dev[dev];
  if (!x.s) {
    SideStream n;
    if (cudaStreamCreateWithFlags(&n.s, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming) != cudaSuccess) {
      if (n.fork) cudaEventDestroy(n.fork);
      cudaStreamDestroy(n.s);
      return false;
    }
    x = n;
  }
  *out = x;
  return true;
}

static int fwd_bwd_impl(const float* delta, const float* u, const float* B, const float* C,
                        const float* gate, const float* A_log, const float* D, const float* dy,
                        float* out, void* ckpt, size_t ckpt_bytes, void* scratch,
                        size_t scratch_bytes, float* d_delta, float* d_u, float* d_B,
                        float* d_C, float* d_A_log, float* d_D, float* d_gate, int64_t batch,
                        int64_t T, int64_t d_inner, int64_t d_state, void* stream, int io_bf16) {
  if (!out) return MAMBA_ERR_INVALID_ARG;
  // everything is checked before the first launch
  int rc = scan_bwd_impl(delta, u, B, C, gate, A_log, D, dy, ckpt, ckpt_bytes, scratch,
                         scratch_bytes, d_delta, d_u, d_B, d_C, d_A_log, d_D, d_gate, batch, T,
                         d_inner, d_state, stream, 0, out, false, true, io_bf16);
  if (rc != MAMBA_OK) return rc;
  Plan plan;
  if (!mscan::make_plan(batch, T, d_inner, d_state, &plan)) return MAMBA_ERR_INVALID_ARG;
  // d_state 9..64 runs the tensor-memory backward. Up to d_state 16 the forward keeps only the
  // checkpoints and the backward forms y and out; above, where forming y costs the backward
  // more than it saves the forward (measured at d_state 64), the forward writes out and y as
  // the separate call does, except with bf16 I/O, whose kernels are the fused ones. Smaller
  // d_state runs the two passes as separate calls do.
  const bool tmem = plan.NP >= mscan::kTmemMinNP;
  const bool fused = tmem && (io_bf16 || plan.NP <= 16);
  // bf16 I/O: the fused path with TMA staging only (16-byte rows of bf16, two chunks or more)
  if (io_bf16 && (!tmem || d_inner % 8 != 0 || d_state % 8 != 0 || plan.nchunks < 2))
    return MAMBA_ERR_UNSUPPORTED;
  // The backward's segment pre-pass and the composition of its carries read only inputs, so in
  // the fused path they run on a side stream beside the forward (which leaves most issue slots
  // idle); the backward proper waits for both. The fork event is recorded before the forward
  // is enqueued, so the forward's CTAs are dispatched first.
  SideStream side;
  const bool overlap = tmem && plan.bwd.nseg > 1 && side_stream(&side);
  const cudaStream_t s = (cudaStream_t)stream;
  if (overlap) {
    if (cudaEventRecord(side.fork, s) != cudaSuccess ||
        cudaStreamWaitEvent(side.s, side.fork, 0) != cudaSuccess)
      return set_cuda_error(cudaGetLastError());
  }
  rc = scan_fwd_impl(delta, u, B, C, gate, A_log, D, out, nullptr, ckpt, ckpt_bytes, batch, T,
                     d_inner, d_state, stream, 0, fused ? 1 : 0, io_bf16);
  if (rc != MAMBA_OK) return rc;
  int launches = g_last_launches;
  if (overlap) {
    rc = scan_bwd_impl(delta, u, B, C, gate, A_log, D, dy, ckpt, ckpt_bytes, scratch,
                       scratch_bytes, d_delta, d_u, d_B, d_C, d_A_log, d_D, d_gate, batch, T,
                       d_inner, d_state, stream, 0, out, fused, false, io_bf16, 1, side.s);
    if (rc == MAMBA_OK) launches += g_last_launches;
    // joined even after a failed launch, so that a captured stream never keeps an open fork
    if (cudaEventRecord(side.join, side.s) != cudaSuccess ||
        cudaStreamWaitEvent(s, side.join, 0) != cudaSuccess)
      return set_cuda_error(cudaGetLastError());
    if (rc != MAMBA_OK) return rc;
  }
  rc = scan_bwd_impl(delta, u, B, C, gate, A_log, D, dy, ckpt, ckpt_bytes, scratch,
                     scratch_bytes, d_delta, d_u, d_B, d_C, d_A_log, d_D, d_gate, batch, T,
                     d_inner, d_state, stream, 0, out, fused, false, io_bf16, overlap ? 2 : 0);
  if (rc != MAMBA_OK) return rc;
  g_last_launches += launches;
  return MAMBA_OK;
}

int mamba_scan_fwd_bwd(const float* delta, const float* u, const float* B, const float* C,
                       const float* gate, const float* A_log, const float* D, const float* dy,
                       float* out, void* ckpt, size_t ckpt_bytes, void* scratch,
                       size_t scratch_bytes, float* d_delta, float* d_u, float* d_B, float* d_C,
                       float* d_A_log, float* d_D, float* d_gate, int64_t batch, int64_t T,
                       int64_t d_inner, int64_t d_state, void* stream) {
  mscan::NvtxRange nvtx_range("mamba_scan_fwd_bwd");
  return fwd_bwd_impl(delta, u, B, C, gate, A_log, D, dy, out, ckpt, ckpt_bytes, scratch,
                      scratch_bytes, d_delta, d_u, d_B, d_C, d_A_log, d_D, d_gate, batch, T,
                      d_inner, d_state, stream, 0);
}

int mamba_scan_fwd_bwd_bf16(const void* delta, const void* u, const void* B, const void* C,
                            const void* gate, const float* A_log, const float* D,
                            const void* dy, void* out, void* ckpt, size_t ckpt_bytes,
                            void* scratch, size_t scratch_bytes, void* d_delta, void* d_u,
                            void* d_B, void* d_C, float* d_A_log, float* d_D, void* d_gate,
                            int64_t batch, int64_t T, int64_t d_inner, int64_t d_state,
                            void* stream) {
  mscan::NvtxRange nvtx_range("mamba_scan_fwd_bwd_bf16");
  // the kernels take the bf16 tensors through the same parameter slots (io_bf16 set)
  auto in = [](const void* q) { return static_cast<const float*>(q); };
  auto io = [](void* q) { return static_cast<float*>(q); };
  return fwd_bwd_impl(in(delta), in(u), in(B), in(C), in(gate), A_log, D, in(dy), io(out), ckpt,
                      ckpt_bytes, scratch, scratch_bytes, io(d_delta), io(d_u), io(d_B), io(d_C),
                      d_A_log, d_D, io(d_gate), batch, T, d_inner, d_state, stream, 1);
}

size_t mamba_scan_host_workspace_bytes(int64_t batch, int64_t T, int64_t d_inner,
                                       int64_t d_state) {
  HostLayout L;
  if (!host_layout(batch, T, d_inner, d_state, &L)) return 0;
  return L.total;
}

// mamba_scan_fwd_bwd_host for a batch smaller than the slice count: slice k is the whole batch
// over channels [k*dcs, k*dcs + dcs) and runs as a scan of its own on its own stream. Its
// inputs come in with 2-D copies (rows of dcs floats out of the host's rows of d_inner), its
// outputs go back the same way, its rows of A_log, D, d_A_log and d_D are plain ranges, and
// d_B, d_C (sums over d_inner) are the slices' sums added in slice order by a small kernel.
static int run_channel_slices(const HostLayout& L, char* w, const float* delta, const float* u,
                              const float* B, const float* C, const float* gate,
                              const float* A_log, const float* D, const float* dy, float* out,
                              float* d_delta, float* d_u, float* d_B, float* d_C,
                              float* d_A_log, float* d_D, float* d_gate, int64_t batch,
                              int64_t T, int64_t d_inner, int64_t d_state, cudaStream_t s0) {
  AuxStreams ax;
  if (!aux_streams(&ax)) return set_cuda_error(cudaGetLastError());
  std::lock_guard<std::mutex> hold(*ax.enqueue);
  ax.s[0] = s0;
  auto at = [&](size_t off) { return (float*)(w + off); };
  const size_t rows = (size_t)batch * T;                 // rows of the [batch*T][d_inner] view
  const size_t btn = rows * (size_t)d_state;             // floats of B (and C)
  float* w_B = at(L.off_bc);
  float* w_C = w_B + btn;
  cudaError_t e;
  // B and C (shared by every slice) first, on the caller's stream
  if ((e = cudaMemcpyAsync(w_B, B, btn * 4, cudaMemcpyHostToDevice, s0)) != cudaSuccess ||
      (e = cudaMemcpyAsync(w_C, C, btn * 4, cudaMemcpyHostToDevice, s0)) != cudaSuccess ||
      (e = cudaEventRecord(ax.ev[kHostSlices], s0)) != cudaSuccess)
    return set_cuda_error(e);
  for (int k = 1; k < L.nslices; ++k)
    if ((e = cudaStreamWaitEvent(ax.s[k], ax.ev[kHostSlices], 0)) != cudaSuccess)
      return set_cuda_error(e);
  int launches = 0;
  const size_t hp = (size_t)d_inner * 4;   // host row pitch
  for (int k = 0; k < L.nslices; ++k) {
    cudaStream_t st = ax.s[k];
    const int64_t d0 = L.sd0[k], nd = L.sdw[k];
    const size_t dp = (size_t)nd * 4;        // device row pitch (compact slice)
    char* sl = w + L.off_slice[k];
    float* in[4];
    float* outv[4];
    for (int i = 0; i < 4; ++i) {
      in[i] = (float*)(sl + L.sl_in[i]);
      outv[i] = (float*)(sl + L.sl_out[i]);
    }
    float* sA = (float*)(sl + L.sl_A);
    float* sD = (float*)(sl + L.sl_D);
    float* sdA = (float*)(sl + L.sl_dA);
    float* sdD = (float*)(sl + L.sl_dD);
    float* part = at(L.off_bcpart) + (size_t)k * 2 * btn;   // d_B | d_C of this slice
    const float* hin[4] = {delta, u, gate, dy};
    // one slice's copies at a time in each direction (slice order), each at the link's rate
    if (k > 0 && (e = cudaStreamWaitEvent(st, ax.ev_in[k - 1], 0)) != cudaSuccess)
      return set_cuda_error(e);
    for (int i = 0; i < 4; ++i)
      if ((e = cudaMemcpy2DAsync(in[i], dp, hin[i] + d0, hp, dp, rows, cudaMemcpyHostToDevice,
                                 st)) != cudaSuccess)
        return set_cuda_error(e);
    if ((e = cudaMemcpyAsync(sA, A_log + (size_t)d0 * d_state, (size_t)nd * d_state * 4,
                             cudaMemcpyHostToDevice, st)) != cudaSuccess ||
        (e = cudaMemcpyAsync(sD, D + d0, dp, cudaMemcpyHostToDevice, st)) != cudaSuccess ||
        (e = cudaEventRecord(ax.ev_in[k], st)) != cudaSuccess)
      return set_cuda_error(e);
    float* ck = at(L.off_ck[k]);
    float* sc = at(L.off_sc[k]);
    int rc = mamba_scan_fwd(in[0], in[1], w_B, w_C, in[2], sA, sD, outv[0], nullptr,
                            L.ck_bytes ? ck : nullptr, L.ck_bytes, batch, T, nd, d_state, st);
    if (rc != MAMBA_OK) return rc;
    launches += g_last_launches;
    if ((e = cudaEventRecord(ax.ev_fwd[k], st)) != cudaSuccess) return set_cuda_error(e);
    rc = mamba_scan_bwd(in[0], in[1], w_B, w_C, in[2], sA, sD, in[3], L.ck_bytes ? ck : nullptr,
                        L.ck_bytes, sc, L.sc_bytes, outv[1], outv[2], part, part + btn, sdA, sdD,
                        outv[3], batch, T, nd, d_state, st);
    if (rc != MAMBA_OK) return rc;
    launches += g_last_launches;
    if ((e = cudaEventRecord(ax.ev_bwd[k], st)) != cudaSuccess) return set_cuda_error(e);
  }
  // The copies out run on the library's device->host stream, one after another in slice order
  // (each at the link's rate), so that the slices' kernels never wait behind them: a slice's out
  // as soon as its forward is done, its gradients once its backward is done. The device->host
  // direction carries as many bytes as the other but can only start after the first slice's
  // forward, so it is the pipeline's critical path.
  cudaStream_t sd = ax.d2h;
  for (int k = 0; k < L.nslices; ++k) {
    const int64_t d0 = L.sd0[k], nd = L.sdw[k];
    const size_t dp = (size_t)nd * 4;
    char* sl = w + L.off_slice[k];
    float* outv[4];
    for (int i = 0; i < 4; ++i) outv[i] = (float*)(sl + L.sl_out[i]);
    float* sdA = (float*)(sl + L.sl_dA);
    float* sdD = (float*)(sl + L.sl_dD);
    float* hout[4] = {out, d_delta, d_u, d_gate};
    if ((e = cudaStreamWaitEvent(sd, ax.ev_fwd[k], 0)) != cudaSuccess ||
        (e = cudaMemcpy2DAsync(hout[0] + d0, hp, outv[0], dp, dp, rows, cudaMemcpyDeviceToHost,
                               sd)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(sd, ax.ev_bwd[k], 0)) != cudaSuccess)
      return set_cuda_error(e);
    for (int i = 1; i < 4; ++i)
      if ((e = cudaMemcpy2DAsync(hout[i] + d0, hp, outv[i], dp, dp, rows, cudaMemcpyDeviceToHost,
                                 sd)) != cudaSuccess)
        return set_cuda_error(e);
    if ((e = cudaMemcpyAsync(d_A_log + (size_t)d0 * d_state, sdA, (size_t)nd * d_state * 4,
                             cudaMemcpyDeviceToHost, sd)) != cudaSuccess ||
        (e = cudaMemcpyAsync(d_D + d0, sdD, dp, cudaMemcpyDeviceToHost, sd)) != cudaSuccess)
      return set_cuda_error(e);
  }
  // d_B and d_C: the slices' sums, added in slice order, then copied out behind the rest
  for (int k = 1; k < L.nslices; ++k)
    if ((e = cudaStreamWaitEvent(s0, ax.ev_bwd[k], 0)) != cudaSuccess) return set_cuda_error(e);
  float* sum = at(L.off_bcsum);
  const size_t n = 2 * btn;
  mscan::sum_slices<<<(unsigned)std::min<size_t>((n + 255) / 256, 65535), 256, 0, s0>>>(
      at(L.off_bcpart), L.nslices, n, sum);
  if ((e = cudaPeekAtLastError()) != cudaSuccess) return set_cuda_error(e);
  ++launches;
  if ((e = cudaEventRecord(ax.ev[0], s0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(sd, ax.ev[0], 0)) != cudaSuccess ||
      (e = cudaMemcpyAsync(d_B, sum, btn * 4, cudaMemcpyDeviceToHost, sd)) != cudaSuccess ||
      (e = cudaMemcpyAsync(d_C, sum + btn, btn * 4, cudaMemcpyDeviceToHost, sd)) != cudaSuccess ||
      (e = cudaEventRecord(ax.ev_end, sd)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(s0, ax.ev_end, 0)) != cudaSuccess)
    return set_cuda_error(e);
  e = cudaStreamSynchronize(s0);
  if (e != cudaSuccess) return set_cuda_error(e);
  g_last_launches = launches;
  if (mscan::bwd_take_fault() | mscan::fwd_take_fault()) return MAMBA_ERR_TIMEOUT;
  if (take_oob()) return MAMBA_ERR_BOUNDS;
  return MAMBA_OK;
}

int mamba_scan_fwd_bwd_host(const float* delta, const float* u, const float* B, const float* C,
                            const float* gate, const float* A_log, const float* D,
                            const float* dy, float* out, float* d_delta, float* d_u, float* d_B,
                            float* d_C, float* d_A_log, float* d_D, float* d_gate,
                            void* workspace, size_t workspace_bytes, int64_t batch, int64_t T,
                            int64_t d_inner, int64_t d_state, void* stream) {
  mscan::NvtxRange nvtx_range("mamba_scan_fwd_bwd_host");
  Plan plan;
  int rc = check_dims(batch, T, d_inner, d_state, &plan);
  if (rc != MAMBA_OK) return rc;
  if (!delta || !u || !B || !C || !gate || !A_log || !D || !dy || !out || !d_delta || !d_u ||
      !d_B || !d_C || !d_A_log || !d_D || !d_gate || !workspace)
    return MAMBA_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return MAMBA_ERR_MISALIGNED;
  HostLayout L;
  if (!host_layout(batch, T, d_inner, d_state, &L)) return MAMBA_ERR_INVALID_ARG;
  if (workspace_bytes < L.total) return MAMBA_ERR_WORKSPACE;
  char* w = (char*)workspace;
  if (L.by_channels)
    return run_channel_slices(L, w, delta, u, B, C, gate, A_log, D, dy, out, d_delta, d_u, d_B,
                              d_C, d_A_log, d_D, d_gate, batch, T, d_inner, d_state,
                              (cudaStream_t)stream);
  auto at = [&](size_t off) { return (float*)(w + off); };
  float *w_delta = at(L.off_in[0]), *w_u = at(L.off_in[1]), *w_gate = at(L.off_in[2]),
        *w_dy = at(L.off_in[3]), *w_B = at(L.off_in[4]), *w_C = at(L.off_in[5]),
        *w_A = at(L.off_in[6]), *w_D = at(L.off_in[7]);
  float *w_out = at(L.off_out[0]), *w_dd = at(L.off_out[1]), *w_du = at(L.off_out[2]),
        *w_dg = at(L.off_out[3]), *w_dB = at(L.off_out[4]), *w_dC = at(L.off_out[5]),
        *w_dA = at(L.off_out[6]), *w_dD = at(L.off_out[7]);
  const size_t td = (size_t)T * d_inner, tn = (size_t)T * d_state;
  const size_t dn = (size_t)d_inner * d_state, dd = (size_t)d_inner;

  // Each slice of the batch runs on its own stream (the caller's for the first, the library's
  // for the others): its copies in, forward, backward and copies out. So the copies in both
  // directions overlap each other and the kernels of other slices.
  cudaStream_t s0 = (cudaStream_t)stream;
  AuxStreams ax;
  if (!aux_streams(&ax)) return set_cuda_error(cudaGetLastError());
  std::lock_guard<std::mutex> hold(*ax.enqueue);
  ax.s[0] = s0;
  auto cp = [&](void* dst, const void* src, size_t n, cudaMemcpyKind k, cudaStream_t st) {
    return cudaMemcpyAsync(dst, src, n, k, st);
  };
  cudaError_t e;
  if ((e = cp(w_A, A_log, dn * 4, cudaMemcpyHostToDevice, s0)) != cudaSuccess ||
      (e = cp(w_D, D, dd * 4, cudaMemcpyHostToDevice, s0)) != cudaSuccess ||
      (e = cudaEventRecord(ax.ev[kHostSlices], s0)) != cudaSuccess)
    return set_cuda_error(e);
  for (int k = 1; k < L.nslices; ++k)
    if ((e = cudaStreamWaitEvent(ax.s[k], ax.ev[kHostSlices], 0)) != cudaSuccess)
      return set_cuda_error(e);
  int launches = 0;
  for (int k = 0; k < L.nslices; ++k) {
    cudaStream_t st = ax.s[k];
    const int64_t b0 = (int64_t)k * L.rows, nb = std::min<int64_t>(L.rows, batch - b0);
    const size_t o_td = (size_t)b0 * td, o_tn = (size_t)b0 * tn;
    const size_t n_td = (size_t)nb * td * 4, n_tn = (size_t)nb * tn * 4;
    float* ck = at(L.off_ck[k]);
    float* sc = at(L.off_sc[k]);
    float* pdA = at(L.off_part) + (size_t)k * (L.dn_pad + L.dd_pad);
    const struct { float* dst; const float* src; size_t n; } in[] = {
        {w_delta + o_td, delta + o_td, n_td}, {w_u + o_td, u + o_td, n_td},
        {w_gate + o_td, gate + o_td, n_td},   {w_dy + o_td, dy + o_td, n_td},
        {w_B + o_tn, B + o_tn, n_tn},         {w_C + o_tn, C + o_tn, n_tn}};
    // one slice's copies at a time in each direction (slice order), each at the link's full
    // rate; the slice's kernels start as soon as its own inputs are in
    if (k > 0 && (e = cudaStreamWaitEvent(st, ax.ev_in[k - 1], 0)) != cudaSuccess)
      return set_cuda_error(e);
    for (const auto& c : in)
      if ((e = cp(c.dst, c.src, c.n, cudaMemcpyHostToDevice, st)) != cudaSuccess)
        return set_cuda_error(e);
    if ((e = cudaEventRecord(ax.ev_in[k], st)) != cudaSuccess) return set_cuda_error(e);
    rc = mamba_scan_fwd(w_delta + o_td, w_u + o_td, w_B + o_tn, w_C + o_tn, w_gate + o_td, w_A,
                        w_D, w_out + o_td, nullptr, L.ck_bytes ? ck : nullptr, L.ck_bytes, nb, T,
                        d_inner, d_state, st);
    if (rc != MAMBA_OK) return rc;
    launches += g_last_launches;
    rc = mamba_scan_bwd(w_delta + o_td, w_u + o_td, w_B + o_tn, w_C + o_tn, w_gate + o_td, w_A,
                        w_D, w_dy + o_td, L.ck_bytes ? ck : nullptr, L.ck_bytes, sc, L.sc_bytes,
                        w_dd + o_td, w_du + o_td, w_dB + o_tn, w_dC + o_tn, pdA, pdA + L.dn_pad,
                        w_dg + o_td, nb, T, d_inner, d_state, st);
    if (rc != MAMBA_OK) return rc;
    launches += g_last_launches;
    const struct { float* dst; const float* src; size_t n; } outs[] = {
        {out + o_td, w_out + o_td, n_td},     {d_delta + o_td, w_dd + o_td, n_td},
        {d_u + o_td, w_du + o_td, n_td},      {d_gate + o_td, w_dg + o_td, n_td},
        {d_B + o_tn, w_dB + o_tn, n_tn},      {d_C + o_tn, w_dC + o_tn, n_tn}};
    if (k > 0 && (e = cudaStreamWaitEvent(st, ax.ev_out[k - 1], 0)) != cudaSuccess)
      return set_cuda_error(e);
    for (const auto& c : outs)
      if ((e = cp(c.dst, c.src, c.n, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return set_cuda_error(e);
    if ((e = cudaEventRecord(ax.ev_out[k], st)) != cudaSuccess) return set_cuda_error(e);
  }
  // d_A_log and d_D: the slices' sums, added in slice order
  for (int k = 1; k < L.nslices; ++k)
    if ((e = cudaEventRecord(ax.ev[k], ax.s[k])) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s0, ax.ev[k], 0)) != cudaSuccess)
      return set_cuda_error(e);
  const size_t npart = L.dn_pad + L.dd_pad;
  mscan::sum_slices<<<(unsigned)((npart + 255) / 256), 256, 0, s0>>>(at(L.off_part), L.nslices,
                                                                      npart, w_dA);
  if ((e = cudaPeekAtLastError()) != cudaSuccess) return set_cuda_error(e);
  ++launches;
  if ((e = cp(d_A_log, w_dA, dn * 4, cudaMemcpyDeviceToHost, s0)) != cudaSuccess ||
      (e = cp(d_D, w_dA + L.dn_pad, dd * 4, cudaMemcpyDeviceToHost, s0)) != cudaSuccess)
    return set_cuda_error(e);
  (void)w_dD;
  e = cudaStreamSynchronize(s0);
  if (e != cudaSuccess) return set_cuda_error(e);
  g_last_launches = launches;
  if (mscan::bwd_take_fault() | mscan::fwd_take_fault()) return MAMBA_ERR_TIMEOUT;
  if (take_oob()) return MAMBA_ERR_BOUNDS;
  return MAMBA_OK;
}

int mamba_scan_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return set_cuda_error(e);
  if (mscan::bwd_take_fault() | mscan::fwd_take_fault()) return MAMBA_ERR_TIMEOUT;
  if (take_oob()) return MAMBA_ERR_BOUNDS;
  return MAMBA_OK;
}

int mamba_scan_bounds_checked(void) {
#ifdef MAMBA_BOUNDS_CHECK
  return 1;
#else
  return 0;
#endif
}

int mamba_scan_test_bounds_shrink(int64_t elements) {
  if (!mamba_scan_bounds_checked()) return MAMBA_ERR_UNSUPPORTED;
  if (elements < 0) return MAMBA_ERR_INVALID_ARG;
  const unsigned long long s = (unsigned long long)elements;
  if (mscan::fwd_set_oob_shrink(s) || mscan::bwd_set_oob_shrink(s) ||
      mscan::tmem_set_oob_shrink(s) || mscan::conv_set_oob_shrink(s))
    return set_cuda_error(cudaGetLastError());
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
    case MAMBA_ERR_BOUNDS:
      return "bounds-checked build: a kernel computed an offset outside its buffer (the access "
             "was not made); recent outputs are invalid";
    default: return "unknown error code";
  }
}

int mamba_scan_last_launch_count(void) { return g_last_launches; }

}  // extern "C"
