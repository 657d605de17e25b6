// C ABI of the conv1d + SiLU step (declared in include/mamba_scan.h): validation, scratch
// sizing and launches.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mamba_scan.h"
#include "conv_plan.h"

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int check(int64_t batch, int64_t T, int64_t Di, int64_t K) {
  if (batch < 1 || T < 1 || Di < 1 || K < 1) return MAMBA_ERR_INVALID_ARG;
  if (K > mscan::kConvMaxK) return MAMBA_ERR_UNSUPPORTED;
  if (batch > 65535 || (double)batch * T * Di >= 2147483648.0) return MAMBA_ERR_INVALID_ARG;
  return MAMBA_OK;
}

size_t scratch_bytes(int64_t batch, int64_t T, int64_t Di, int64_t K) {
  const size_t a = 64;   // floats: 256-byte regions
  const size_t w = (mscan::conv_part_w_floats(batch, T, Di, K) + a - 1) / a * a;
  const size_t b = (mscan::conv_part_b_floats(batch, T, Di) + a - 1) / a * a;
  return (w + b) * sizeof(float);
}

}  // namespace

extern "C" {

size_t mamba_conv_scratch_bytes(int64_t batch, int64_t T, int64_t d_inner, int64_t d_conv) {
  if (check(batch, T, d_inner, d_conv) != MAMBA_OK) return 0;
  return scratch_bytes(batch, T, d_inner, d_conv);
}

int mamba_conv_fwd(const float* x, const float* w, const float* bias, float* u, int64_t batch,
                   int64_t T, int64_t d_inner, int64_t d_conv, void* stream) {
  int rc = check(batch, T, d_inner, d_conv);
  if (rc != MAMBA_OK) return rc;
  if (!x || !w || !bias || !u) return MAMBA_ERR_INVALID_ARG;
  const void* ptrs[] = {x, w, bias, u};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MAMBA_ERR_MISALIGNED;
  const size_t n = (size_t)batch * T * d_inner * sizeof(float);
  if ((uintptr_t)u < (uintptr_t)x + n && (uintptr_t)x < (uintptr_t)u + n)
    return MAMBA_ERR_INVALID_ARG;   // u must not overlap x
  mscan::ConvParams p = {};
  p.x = x; p.w = w; p.bias = bias; p.u = u;
  p.batch = (int)batch; p.T = (int)T; p.Di = (int)d_inner; p.K = (int)d_conv;
  p.run = mscan::kConvRun;   // the launch picks the run length
  p.nruns = mscan::conv_nruns(T);
  p.ngroups = mscan::conv_ngroups(T);
  const int k = mscan::launch_conv(p, false, (cudaStream_t)stream);
  if (k < 0) return MAMBA_ERR_CUDA;
  return MAMBA_OK;
}

int mamba_conv_bwd(const float* x, const float* w, const float* bias, const float* d_u,
                   void* scratch, size_t scratch_bytes_, float* d_x, float* d_w, float* d_bias,
                   int64_t batch, int64_t T, int64_t d_inner, int64_t d_conv, void* stream) {
  int rc = check(batch, T, d_inner, d_conv);
  if (rc != MAMBA_OK) return rc;
  if (!x || !w || !bias || !d_u || !scratch || !d_x || !d_w || !d_bias)
    return MAMBA_ERR_INVALID_ARG;
  const void* ptrs[] = {x, w, bias, d_u, scratch, d_x, d_w, d_bias};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MAMBA_ERR_MISALIGNED;
  if (scratch_bytes_ < scratch_bytes(batch, T, d_inner, d_conv)) return MAMBA_ERR_WORKSPACE;
  const size_t n = (size_t)batch * T * d_inner * sizeof(float);
  auto ov = [](const void* a, size_t na, const void* b, size_t nb) {
    return (uintptr_t)a < (uintptr_t)b + nb && (uintptr_t)b < (uintptr_t)a + na;
  };
  const size_t nw = (size_t)d_inner * d_conv * sizeof(float), nb = (size_t)d_inner * 4;
  const size_t ns = scratch_bytes(batch, T, d_inner, d_conv);
  if (ov(d_x, n, x, n) || ov(d_x, n, d_u, n) || ov(d_x, n, scratch, ns) || ov(d_w, nw, scratch, ns) ||
      ov(d_bias, nb, scratch, ns) || ov(d_x, n, d_w, nw) || ov(d_x, n, d_bias, nb) ||
      ov(d_w, nw, d_bias, nb))
    return MAMBA_ERR_INVALID_ARG;
  mscan::ConvParams p = {};
  p.x = x; p.w = w; p.bias = bias; p.d_u = d_u;
  p.d_x = d_x; p.d_w = d_w; p.d_bias = d_bias;
  float* sc = (float*)scratch;
  const size_t a = 64;
  p.part_w = sc;
  p.part_b = sc + (mscan::conv_part_w_floats(batch, T, d_inner, d_conv) + a - 1) / a * a;
  p.batch = (int)batch; p.T = (int)T; p.Di = (int)d_inner; p.K = (int)d_conv;
  p.run = mscan::kConvRun;   // the launch picks the run length
  p.nruns = mscan::conv_nruns(T);
  p.ngroups = mscan::conv_ngroups(T);
  const int k = mscan::launch_conv(p, true, (cudaStream_t)stream);
  if (k < 0) return MAMBA_ERR_CUDA;
  return MAMBA_OK;
}

}  // extern "C"
