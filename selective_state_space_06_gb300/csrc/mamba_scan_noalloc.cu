// mamba_scan_bwd_noalloc: the backward scan for callers that cannot allocate device memory.
//
// Some callers get only their input and output buffers, and must not allocate device memory
// themselves, not even through the caller-sized scratch argument of mamba_scan_bwd. Two
// examples: a plugin running inside a host framework that owns every byte of device memory,
// and a latency-critical loop that forbids cudaMalloc, which can synchronise the whole device.
// For them, this entry point takes the backward's scratch from a fixed file-scope device array
// instead of from the caller.
//
// How it works. g_noalloc_scratch is a static __device__ array of
// MAMBA_SCAN_NOALLOC_SCRATCH_BYTES. Every GPU that loads the library holds it until the
// process exits. In host code the array's name is only a host-side stand-in, not a device
// address. So the first call on each device, with that device current, asks the runtime for the
// array's device address (cudaGetSymbolAddress), checks the result and caches it. Every later
// call on that device reuses the cached address. Because the first call does this set-up, it
// should come before any stream capture. The call itself allocates nothing: no cudaMalloc, no
// cudaFree, no allocating library routine.
//
// Sharing. All calls on a device share the one array, and it keeps the last call's contents.
// The backward writes every scratch word it later reads (its per-CTA partial sums), so nothing
// has to be cleared between calls. Calls that overlap on the GPU (different streams, or
// different host threads without ordering) race on the array and give wrong results: the caller
// must order them.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mamba_scan.h"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[MAMBA_SCAN_NOALLOC_SCRATCH_BYTES];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (set up once per device).
int noalloc_scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MAMBA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MAMBA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MAMBA_OK;
}

}  // namespace

extern "C" int mamba_scan_bwd_noalloc(const float* delta, const float* u, const float* B,
                                      const float* C, const float* gate, const float* A_log,
                                      const float* D, const float* dy, const void* ckpt,
                                      size_t ckpt_bytes, float* d_delta, float* d_u, float* d_B,
                                      float* d_C, float* d_A_log, float* d_D, float* d_gate,
                                      int64_t batch, int64_t T, int64_t d_inner, int64_t d_state,
                                      void* stream) {
  const size_t need = mamba_scan_scratch_bytes(batch, T, d_inner, d_state);
  if (need == 0) {
    // sizes invalid: let the regular entry point name the error (it launches nothing then)
    return mamba_scan_bwd(delta, u, B, C, gate, A_log, D, dy, ckpt, ckpt_bytes, nullptr, 0,
                          d_delta, d_u, d_B, d_C, d_A_log, d_D, d_gate, batch, T, d_inner,
                          d_state, stream);
  }
  if (need > (size_t)MAMBA_SCAN_NOALLOC_SCRATCH_BYTES) return MAMBA_ERR_NOALLOC_LIMIT;
  void* scratch = nullptr;
  const int rc = noalloc_scratch_address(&scratch);
  if (rc != MAMBA_OK) return rc;
  return mamba_scan_bwd(delta, u, B, C, gate, A_log, D, dy, ckpt, ckpt_bytes, scratch,
                        (size_t)MAMBA_SCAN_NOALLOC_SCRATCH_BYTES, d_delta, d_u, d_B, d_C, d_A_log,
                        d_D, d_gate, batch, T, d_inner, d_state, stream);
}
