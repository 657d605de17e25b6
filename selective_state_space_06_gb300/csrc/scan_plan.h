// Internal (not part of the C ABI): launch plan and kernel parameter blocks shared by the
// host entry points (mamba_scan_abi.cu) and the kernel launchers (scan_fwd.cu, scan_bwd.cu).
#pragma once
#include <cuda.h>   // CUtensorMap (the type only)
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mscan {

// Thread mapping of both scan kernels (see scan_fwd.cu for the picture):
//   a thread owns kDPT consecutive channels d and NPT = states_per_thread(NP) consecutive
//   states n; G = NP / NPT lanes of a warp share the same channels and split the states
//   between them; a warp therefore covers (32 / G) * kDPT channels; a CTA has kWarps warps.
constexpr int kDPT = 2;     // channels per thread
// States per thread (2 or 4) for d_state padded to NP. Measured on GB300: the forward is
// fastest with 2 states per thread up to d_state 16 (twice the threads, so more latency hiding)
// and with 4 beyond; the backward is fastest with 4 (fewer cross-lane reductions per element).
__host__ __device__ constexpr int states_per_thread_fwd(int NP) { return NP <= 16 ? 2 : 4; }
__host__ __device__ constexpr int states_per_thread_bwd(int NP) { return NP < 4 ? NP : 4; }
// Channels per thread of the forward kernels (2 or 4). Each thread loads the B and C values of
// its states once per step for all of its channels, so more channels per thread deliver fewer
// shared-memory bytes per (element, state). Measured on GB300: 4 at d_state 64 (longseq
// forward 4.53 -> 4.18 ms, where the kernel is bound by the shared-memory data path), 2 below
// (4 at d_state 16 is slower: half the warps, mamba130m forward 0.111 -> 0.138 ms).
__host__ __device__ constexpr int fwd_channels_per_thread(int NP) { return NP == 64 ? 4 : 2; }
constexpr int kWarps = 4;   // warps per CTA
// Warps per CTA of the forward scan. Measured on GB300: at d_state 16, where the forward has no
// time segments and its CTAs are as many as the batch rows x channel blocks (512 at mamba370m,
// 3.4 per SM), 2 warps per CTA (twice the CTAs, spread more evenly) took 0.230 ms at mamba370m
// and 0.093 at mamba130m against 0.240 and 0.098 with 4, and 1 warp 0.257 and 0.104. At d_state
// 64 (segments filling whole waves) 4 warps are best: longseq's forward took 3.66 ms, against
// 3.74 with 2 and 4.45 with 1.
__host__ __device__ constexpr int fwd_warps(int NP) { return NP <= 16 ? 2 : 4; }
// Warps per CTA of the backward pre-pass at d_state <= 8 (the main kernel's CTA shape measured
// best; wider CTAs with several segments each were slower on GB300).
constexpr int kAggWarps = kWarps;
constexpr int kSMs = 152;   // GB300
// Resident CTAs per SM of the backward pre-pass of the tensor-memory path
// (scan_bwd_agg4_kernel): 4 at d_state 16 (its two stages take 51 KB of shared memory), 7 at
// d_state 32 and 64 (70 registers per thread). Its sub-segments are chosen to fill whole waves
// of them. Measured on GB300 at the long-sequence layer: the backward call took 8.69 ms with 8
// sub-segments per segment (11 waves), 8.70 with 2 (3 waves) and 8.80 with 1 (1440 CTAs, 1.35
// waves: the earlier fixed target of 1216 CTAs).
__host__ __device__ constexpr int bwd_agg_ctas_per_sm(int NP) { return NP <= 16 ? 4 : 7; }
constexpr int kChunk = 16;  // time steps per chunk (= checkpoint interval)
constexpr int kMaxState = 64;

// The time axis is cut into nseg segments of seg_chunks chunks. One CTA handles one unit
// (batch row, block of DC channels, segment). The state entering a segment comes from a small
// pre-pass kernel that scans every segment independently from zero (the forward's aggregates:
// the local end state and the sum of delta). For the backward, the pre-pass gives the local
// d_h prefix and the sum of delta. The linear recurrence composes these aggregates exactly, so
// the segments run in parallel.
// Units (CTAs) to aim for per pass. The forward segments the time axis only at d_state > 16:
// below that its pre-pass costs more than the extra parallelism gains (measured on GB300).
__host__ __device__ constexpr int target_units_fwd(int NP) { return NP <= 16 ? 1 : 2048; }
__host__ __device__ constexpr int target_units_bwd(int NP) { return 2048; }
// At d_state 64 the forward (tensor copies, 3 stages) keeps 5 CTAs per SM, and its segments are
// chosen so that its CTAs fill kFwdWaves64 whole waves of them (as nearly as the batch rows x
// channel blocks allow). Measured at the long-sequence layer (80 channel blocks) on GB300, with
// the segments' start states composed by a kernel of their own: the forward call took 3.66 ms
// with 76 segments (8 waves), 3.67 with 57 (6) or 114 (12), 3.68 with 152 (16) and 3.69 with 38
// (4). (When each CTA composed the aggregates of all earlier segments itself, that cost grew
// with the segment count, and 38 segments were best at 3.72 ms; a fixed target of 2048 CTAs,
// 26 segments and 2.7 waves, took 3.83 ms.)
constexpr int kFwdSlots64 = 5 * 152;
constexpr int kFwdWaves64 = 8;
// The backward for d_state > 8 runs scan_bwd_tmem_kernel: 4 channels x 4 states per thread,
// at most 2 CTAs per SM (its tensor-memory columns), so its segments are chosen to fill whole
// waves of 2 x 152 CTAs.
constexpr int kTmemMinNP = 16;
constexpr int kTmemDPT = 4;
constexpr int kTmemSlots = 2 * 152;

// Work decomposition of one pass (forward or backward); the two may differ.
struct PassPlan {
  int NPT = 0;         // states per thread
  int G = 0;           // lanes per channel group
  int DC = 0;          // channels per CTA
  int nblk = 0;        // CTAs along d_inner
  int seg_chunks = 0;  // chunks per segment
  int nseg = 0;        // segments along T
  // backward only: the segment pre-pass works on sub-segments of sub_chunks chunks (nsub per
  // segment, the last ones possibly shorter or empty), so that it has enough CTAs even when
  // the main kernel wants few, long segments
  int sub_chunks = 0;
  int nsub = 1;
};

struct Plan {
  int64_t batch = 0, T = 0, Di = 0, N = 0;
  int NP = 0;          // d_state padded to 4, 8, 16, 32 or 64
  int nchunks = 0;     // chunks along T
  PassPlan fwd, bwd;
  // checkpoint buffer layout (float offsets, 256-byte aligned regions):
  //   [batch][nchunks-1][Di][N] chunk-boundary states, then the forward aggregates
  //   [batch][fwd.nseg][Di][N] segment end states (from zero) and [batch][fwd.nseg][Di] sums
  //   of delta
  //   and y [batch][T][Di], which the backward needs for d_gate
  size_t off_fagg_h = 0, off_fagg_sd = 0, off_y = 0, ckpt_elems = 0;
  // scratch layout (float offsets, each region 256-byte aligned)
  size_t off_partB = 0, off_partC = 0, off_partA = 0, off_partD = 0;
  size_t off_bagg_L = 0, off_bagg_sd = 0, scratch_elems = 0;
};

// Records a CUDA error as the one mamba_scan_strerror(MAMBA_ERR_CUDA) reports, and returns
// MAMBA_ERR_CUDA (for entry points outside mamba_scan_abi.cu).
int record_cuda_error(cudaError_t e);

// Returns false when the sizes are outside what the kernels support (scan_plan.cu).
bool make_plan(int64_t batch, int64_t T, int64_t Di, int64_t N, Plan* plan);
// x rounded up to a multiple of a
size_t round_up(size_t x, size_t a);

struct FwdParams {
  const float* delta; const float* u; const float* B; const float* C; const float* gate;
  const float* A_log; const float* D;
  float* out; float* y; float* ckpt;
  float* agg_h; float* agg_sd;   // forward segment aggregates (inside the ckpt buffer)
  float* y_ck;                   // y = sum_n C*h + D*u for the backward (inside the ckpt buffer)
  int batch, T, Di, N, nchunks, nblk, seg_chunks, nseg;
  int agg_k;                     // pre-pass: consecutive segments per CTA
  int softplus;                  // delta holds the raw delta: the kernels apply softplus
  int states_only;               // checkpoints only: no C, gate reads, no out, y (fused call)
  int io_bf16;                   // delta, u, B point at bf16 data (states-only forward)
  // Failure-path test only (mamba_scan_fwd_test_timeout): the forward kernel with tensor
  // copies (d_state 64) issues no copy for the last chunk of each CTA, so the wait for it runs
  // out after wait_limit_ns.
  int test_skip_last_copy;
  unsigned long long wait_limit_ns;   // bound of every copy wait of the forward (0: one second)
  // buffer lengths in elements, for the bounds-checked build
  __host__ __device__ size_t n_io() const { return (size_t)batch * T * Di; }
  __host__ __device__ size_t n_bc() const { return (size_t)batch * T * N; }
  __host__ __device__ size_t n_ck() const { return (size_t)batch * (nchunks - 1) * Di * N; }
  __host__ __device__ size_t n_agg_h() const { return (size_t)batch * nseg * Di * N; }
  __host__ __device__ size_t n_agg_sd() const { return (size_t)batch * nseg * Di; }
};

struct BwdParams {
  const float* delta; const float* u; const float* B; const float* C; const float* gate;
  const float* A_log; const float* D; const float* dy; const float* ckpt;
  const float* y_ck;   // y saved by the forward (inside the ckpt buffer)
  float* d_delta; float* d_u; float* d_gate;
  float* partB; float* partC; float* partA; float* partD;   // scratch
  float* agg_L; float* agg_sd;     // scratch: backward aggregates [batch][nseg*nsub][Di](N)
  float* d_B; float* d_C; float* d_A_log; float* d_D;
  int batch, T, Di, N, nchunks, nblk, seg_chunks, nseg;
  int sub_chunks, nsub;            // pre-pass sub-segments (see PassPlan)
  int softplus;                    // delta holds the raw delta; d_delta receives d_raw
  float* out;   // fused call: the backward recomputes y from the states and writes out (y_ck
                // unused); null otherwise
  int io_bf16;  // fused call only: delta, u, B, C, gate, dy, out, d_delta, d_u, d_B, d_C,
                // d_gate point at bf16 data (A_log, D, d_A_log, d_D stay fp32)
  // Failure-path test only (mamba_scan_bwd_test_timeout): the tensor-memory backward issues no
  // copy for the last chunk of each CTA, so the wait for it runs out after wait_limit_ns.
  int test_skip_last_copy;
  unsigned long long wait_limit_ns;   // bound of every copy wait of the backward's kernels
  // buffer lengths in elements, for the bounds-checked build
  __host__ __device__ size_t n_io() const { return (size_t)batch * T * Di; }
  __host__ __device__ size_t n_bc() const { return (size_t)batch * T * N; }
  __host__ __device__ size_t n_ck() const { return (size_t)batch * (nchunks - 1) * Di * N; }
  __host__ __device__ size_t n_part_bc() const { return (size_t)nblk * batch * T * N; }
  __host__ __device__ size_t n_part_a() const { return (size_t)batch * nseg * Di * N; }
  __host__ __device__ size_t n_part_d() const { return (size_t)batch * nseg * Di; }
  __host__ __device__ size_t n_agg_l() const { return (size_t)batch * nseg * nsub * Di * N; }
  __host__ __device__ size_t n_agg_sd() const { return (size_t)batch * nseg * nsub * Di; }
};

// Encodes a tiled tensor map (no interleave, no swizzle, zero fill outside the tensor) through
// the driver entry point; false when the driver or the arguments refuse it.
bool encode_tiled(CUtensorMap* m, CUtensorMapDataType ty, const void* base, cuuint32_t rank,
                  const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box);

// TMA descriptors of the tensor-memory backward, encoded on the host for each call:
// delta, u, gate, dy, y as [batch][T][d_inner] with boxes of 16 steps x DC channels; B, C as
// [batch][T][d_state] with boxes of 16 steps x NP states; the checkpoints as
// [batch][chunk][d_inner][d_state] with boxes of DC channels x NP states.
struct BwdMaps {   // each CUtensorMap carries its own 64-byte alignment
  CUtensorMap delta, u, gate, dy, y, B, C, ckpt;
};

// TMA descriptors of the forward kernels (d_state 64, d_inner a multiple of 4, fp32 inputs):
// delta, u, gate as [batch][T][d_inner] with boxes of 16 steps x DC channels;
// B, C as [batch][T][d_state] with boxes of 16 steps x NP states. Maps of tensors a variant
// does not read are encoded on delta or B and never used.
struct FwdMaps {
  CUtensorMap delta, u, gate, B, C;
};

// Reads and clears the fault word that the backward kernels set when a bounded wait on an
// asynchronous copy gave up (0: none). Synchronises with the device.
unsigned bwd_take_fault();
// The same for the forward kernels' copy waits.
unsigned fwd_take_fault();
// Fault words of the bounds-checked build, one per kernel file (scan_common.cuh,
// MSCAN_OOB_HOOKS): take returns the word and clears it; set_oob_shrink sets the test hook and
// returns -1 in the default build.
unsigned int fwd_take_oob();
unsigned int bwd_take_oob();
unsigned int tmem_take_oob();
unsigned int conv_take_oob();
int fwd_set_oob_shrink(unsigned long long s);
int bwd_set_oob_shrink(unsigned long long s);
int tmem_set_oob_shrink(unsigned long long s);
int conv_set_oob_shrink(unsigned long long s);

// Each returns the number of kernels enqueued (>= 1) or -1 on a launch error.
// launch_fwd enqueues the segment pre-pass and the composition of its aggregates (when
// nseg > 1) and the forward scan; launch_bwd
// enqueues the backward pre-pass (when nseg > 1), the backward scan and the fixed-order
// reduction.
int launch_fwd(const Plan& plan, const FwdParams& p, cudaStream_t stream);
int launch_bwd(const Plan& plan, const BwdParams& p, cudaStream_t stream);
// the main backward kernel alone for d_state padded to 16, 32 or 64 (scan_bwd_tmem.cu)
int launch_bwd_main_tmem(const Plan& plan, const BwdParams& p, cudaStream_t stream);
// its segment pre-pass (0 kernels when there is one segment)
int launch_bwd_agg_tmem(const Plan& plan, const BwdParams& p, cudaStream_t stream);
// launch_bwd split in two for d_state 9..64: the pre-pass and the composition of the carries
// (inputs only), then the backward and the reduction
int launch_bwd_carries(const Plan& plan, const BwdParams& p, cudaStream_t stream);
int launch_bwd_after_carries(const Plan& plan, const BwdParams& p, cudaStream_t stream);

}  // namespace mscan
