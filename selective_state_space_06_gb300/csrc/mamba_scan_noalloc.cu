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
// array's device address (cudaGetSymbolAddress), checks the result and caches it together with
// the identity of the CUDA context it belongs to (cuCtxGetId). A later call in the same context
// reuses the address; a call in another context (a new primary context after cudaDeviceReset,
// or a context the caller made current) looks it up again. Because the first call in a context
// does this set-up, it should come before any stream capture. A failed look-up returns
// MAMBA_ERR_CUDA with the CUDA error recorded for mamba_scan_strerror. The call itself allocates
// nothing: no cudaMalloc, no cudaFree, no allocating library routine.
//
// Sharing. All calls on a device share the one array, and it keeps the last call's contents.
// The backward writes every scratch word it later reads (its per-CTA partial sums), so nothing
// has to be cleared between calls. Calls that overlap on the GPU (different streams, or
// different host threads without ordering) race on the array and give wrong results: the caller
// must order them.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mamba_scan.h"
#include "scan_plan.h"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[MAMBA_SCAN_NOALLOC_SCRATCH_BYTES];

// The CUDA driver API's context queries, looked up once through the runtime (no driver library
// linked).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
struct CtxFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};
const CtxFns& ctx_fns() {
  static CtxFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return f;
}

// Identity of the current context (0 when it cannot be told, or no context is current yet).
unsigned long long current_context_id() {
  const CtxFns& f = ctx_fns();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!f.get_current || !f.get_id || f.get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (f.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

// Device address of g_noalloc_scratch in the current context of the current device.
int noalloc_scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return mscan::record_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return mscan::record_cuda_error(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  const unsigned long long ctx = current_context_id();
  if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return mscan::record_cuda_error(e);
    if (!p) return mscan::record_cuda_error(cudaErrorInvalidSymbol);
    g_scratch_addr[dev] = p;
    // the look-up makes the device's primary context current when none was
    g_scratch_ctx[dev] = ctx ? ctx : current_context_id();
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
