// Launch plan of the scan kernels: the work decomposition of each pass (threads per channel
// group, channels per CTA, time segments) and the layouts of the checkpoint and scratch
// buffers, from the sizes alone.
#include <algorithm>

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
  auto pass = [&](int npt, int dpt, int warps = kWarps) {
    PassPlan q;
    q.NPT = npt;
    q.G = p.NP / npt;
    q.DC = warps * (32 / q.G) * dpt;
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
  {
    const PassPlan q =
        pass(states_per_thread_fwd(p.NP), fwd_channels_per_thread(p.NP), fwd_warps(p.NP));
    const int64_t rows = (int64_t)batch * q.nblk;
    // d_state 64: the most segments whose CTAs fit in kFwdWaves64 waves (at least one segment)
    const int64_t target =
        p.NP == 64 ? std::max<int64_t>(1, (int64_t)kFwdWaves64 * kFwdSlots64 / rows) * rows
                   : (int64_t)target_units_fwd(p.NP);
    p.fwd = by_target(q, (int)std::min<int64_t>(target, INT32_MAX));
  }
  if (p.NP >= kTmemMinNP)
    p.bwd = by_waves(pass(4, kTmemDPT), kTmemSlots);
  else
    p.bwd = by_target(pass(states_per_thread_bwd(p.NP), kDPT), target_units_bwd(p.NP));
  p.bwd.sub_chunks = p.bwd.seg_chunks;
  p.bwd.nsub = 1;
  if (p.NP >= kTmemMinNP && p.bwd.nseg > 1) {
    // pre-pass CTAs: batch x (the main kernel's channel blocks) x (segments 1 .. nseg-1) x nsub
    // k sub-segments per segment: the fewest chunk steps on the critical path, counted as
    // whole waves of resident pre-pass CTAs times (chunks per sub-segment + 2 of start-up)
    const int64_t base = (int64_t)batch * p.bwd.nblk * (p.bwd.nseg - 1);
    const int64_t slots = (int64_t)bwd_agg_ctas_per_sm(p.NP) * kSMs;
    int64_t k = 1;
    double best = 1e300;
    // (at most 1024 sub-segments a segment: bounds the search, and the carries' composition)
    for (int64_t kk = 1; kk <= std::min<int64_t>(p.bwd.seg_chunks, 1024); ++kk) {
      const int64_t sub = (p.bwd.seg_chunks + kk - 1) / kk;
      const double cost = (double)((base * kk + slots - 1) / slots) * (double)(sub + 2);
      if (cost < best - 1e-9) { best = cost; k = kk; }
    }
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

