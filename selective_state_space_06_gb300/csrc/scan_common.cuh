// Device helpers shared by the scan kernels.
#pragma once
#include <cuda.h>   // CUtensorMap (the type only; no driver library is linked)
#include <cuda_runtime.h>
#include <stdint.h>

#include "scan_plan.h"

namespace mscan {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)
constexpr float kLn2 = 0.6931471805599453f;    // ln(2)
constexpr unsigned kFull = 0xffffffffu;

// ---- bounds-checked builds -------------------------------------------------------------------
// Built with -DMAMBA_BOUNDS_CHECK, every global access whose offset a kernel computes is first
// checked against the length of its buffer (elements, from the sizes the launch carries). An
// access outside is not made: a load reads zero, a store is dropped, and the translation
// unit's fault word records it (mamba_scan_status then reports MAMBA_ERR_BOUNDS). The test hook
// g_oob_shrink takes every length that many elements smaller, so a test can watch the check
// fire on the last elements of each buffer while every access it blocks is still in bounds.
// Without the macro inb() is the constant true and every check compiles away.
#ifdef MAMBA_BOUNDS_CHECK
static __device__ unsigned int g_oob;
static __device__ unsigned long long g_oob_shrink;
// elements [off, off + n) lie inside the first len - shrink elements
__device__ __forceinline__ bool inb(size_t off, size_t n, size_t len) {
  const size_t s = (size_t)g_oob_shrink;
  if (off + n <= len && len - (off + n) >= s) return true;
  atomicOr(&g_oob, 1u);
  return false;
}
// host side of this translation unit's fault word: name##_take_oob() returns it and clears it,
// name##_set_oob_shrink() sets the test hook
#define MSCAN_OOB_HOOKS(name)                                                       \
  unsigned int name##_take_oob() {                                                  \
    unsigned int v = 0;                                                             \
    if (cudaMemcpyFromSymbol(&v, g_oob, sizeof(v)) != cudaSuccess) return 0;        \
    if (v) {                                                                        \
      const unsigned int zero = 0;                                                  \
      cudaMemcpyToSymbol(g_oob, &zero, sizeof(zero));                               \
    }                                                                               \
    return v;                                                                       \
  }                                                                                 \
  int name##_set_oob_shrink(unsigned long long s) {                                 \
    return cudaMemcpyToSymbol(g_oob_shrink, &s, sizeof(s)) == cudaSuccess ? 0 : -1; \
  }
#else
__device__ __forceinline__ constexpr bool inb(size_t, size_t, size_t) { return true; }
#define MSCAN_OOB_HOOKS(name)                                      \
  unsigned int name##_take_oob() { return 0; }                     \
  int name##_set_oob_shrink(unsigned long long) { return -1; }
#endif


// 2^x on the special-function unit (PTX ex2.approx.ftz.f32). In the scan x <= 0, so the result
// lies in [0, 1]; very negative x flushes to 0.
__device__ __forceinline__ float ex2_sfu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// sigmoid(g) = 1 / (1 + 2^(-g*log2 e)). For g << 0 the denominator overflows to +inf and the
// quotient is 0; for g >> 0 it is 1.
__device__ __forceinline__ float sigmoid_fast(float g) {
  return __fdividef(1.0f, 1.0f + ex2_sfu(-g * kLog2e));
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Packed fp32x2 arithmetic (one issue slot for two lanes of work on sm_100+).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }
__device__ __forceinline__ float2 ex2_2(float2 x) { return make_float2(ex2_sfu(x.x), ex2_sfu(x.y)); }

// Shared-memory loads of the staged tiles, as volatile asm. The step loops are fully unrolled
// so that the register stash is statically indexed. With plain loads the compiler hoists the
// loads of many future steps and runs out of registers. Volatile loads stay in program order
// among themselves, while the arithmetic, shuffles and stores around them may still overlap
// neighbouring steps. The tiles are written by cp.async and published by __syncthreads, so no
// ordering inside a thread is lost.
__device__ __forceinline__ float lds1(const float* p) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(smem_addr(p)));
  return v;
}
__device__ __forceinline__ float2 lds2(const float* p) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(smem_addr(p)));
  return v;
}
__device__ __forceinline__ float4 lds4(const float* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

// Predicated stores without a branch. A conditional store inside the unrolled step loops would
// split them into basic blocks and stop the scheduler from overlapping neighbouring steps. When
// the predicate is false the address is never accessed, so it may point past the buffer.
__device__ __forceinline__ void st_global_if(float* p, float v, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.global.f32 [%0], %1;\n\t}"
      ::"l"(p), "f"(v), "r"((unsigned)pred) : "memory");
}
__device__ __forceinline__ void st_shared_if(float* p, float v, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.shared.f32 [%0], %1;\n\t}"
      ::"r"(smem_addr(p)), "f"(v), "r"((unsigned)pred) : "memory");
}

// Predicated store "if (a < b) *p = v" without a branch.
__device__ __forceinline__ void st_global_lt(float* p, float v, int a, int b) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.lt.s32 q, %2, %3;\n\t@q st.global.f32 [%0], %1;\n\t}"
      ::"l"(p), "f"(v), "r"(a), "r"(b) : "memory");
}

// Softplus of the raw delta with the threshold 20 (the identity above it), and its derivative
// (the logistic sigmoid; 1 above the threshold), as in the Softplus backward step of mamba-rs
// src/mamba_ssm/cpu/backward.rs.
// On the SFU: e = 2^(x log2 e), log(1 + e) = log2(1 + e) ln 2. Below e = 2^-10 the rounding of
// 1 + e would cost relative accuracy, and the series e (1 - e/2) is used instead (relative
// error below e^2/3 < 4e-7); above it log2 near 1 is accurate to about 2^-22 absolute, a
// relative error below 4e-6 of log(1 + e) >= 9.7e-4.
__device__ __forceinline__ float log1p_of_exp(float e) {
  return e > 0x1p-10f ? __log2f(1.f + e) * kLn2 : e * fmaf(-0.5f, e, 1.f);
}
__device__ __forceinline__ float softplus_f(float x) {
  return x > 20.f ? x : log1p_of_exp(ex2_sfu(x * kLog2e));
}
// Both at once from one e^x; the derivative is e / (1 + e).
__device__ __forceinline__ void softplus_both(float x, float& sp, float& grad) {
  const float e = ex2_sfu(x * kLog2e);
  sp = x > 20.f ? x : log1p_of_exp(e);
  grad = x > 20.f ? 1.f : __fdividef(e, 1.f + e);
}
// In place over a staged [kChunk][TW] tile of raw delta: rows at or past rows_valid and columns
// at or past cols_valid stay zero (zero delta is an exact no-op of the recurrences).
template <int TW, int NTH>
__device__ __forceinline__ void softplus_tile(float* tile, int rows_valid, int cols_valid) {
  for (int e = threadIdx.x; e < kChunk * TW; e += NTH) {
    const int i = e / TW, col = e % TW;
    if (i < rows_valid && col < cols_valid) tile[e] = softplus_f(tile[e]);
  }
}

// Compiler-level fence between the steps of a fully unrolled loop: no memory access moves
// across it, so the loads of later steps are not hoisted (and kept live in registers) early.
__device__ __forceinline__ void step_fence() { asm volatile("" ::: "memory"); }

// NPR float2 pairs of consecutive states from shared memory (8- or 16-byte aligned).
template <int NPR>
__device__ __forceinline__ void lds_pairs(const float* p, float2 (&out)[NPR]) {
  static_assert(NPR == 1 || NPR == 2 || NPR == 4, "2, 4 or 8 states per thread");
  if constexpr (NPR == 1) {
    out[0] = lds2(p);
  } else {
#pragma unroll
    for (int k = 0; k < NPR / 2; ++k) {
      const float4 v = lds4(p + 4 * k);
      out[2 * k] = make_float2(v.x, v.y);
      out[2 * k + 1] = make_float2(v.z, v.w);
    }
  }
}
// NPR float2 pairs to global memory with 16-byte vector stores (one 8-byte store for NPR 1).
template <int NPR>
__device__ __forceinline__ void st_pairs(float* p, const float2 (&v)[NPR]) {
  if constexpr (NPR == 1) {
    *reinterpret_cast<float2*>(p) = v[0];
  } else {
#pragma unroll
    for (int k = 0; k < NPR / 2; ++k)
      *reinterpret_cast<float4*>(p + 4 * k) =
          make_float4(v[2 * k].x, v[2 * k].y, v[2 * k + 1].x, v[2 * k + 1].y);
  }
}
// The same for the states n0 .. n0+2*NPR-1 of a row of N states (N % 4 == 0, n0 % 4 == 0):
// only the groups of four inside the row are stored; loads give zeros past it.
template <int NPR>
__device__ __forceinline__ void st_pairs_row(float* row, int n0, int N, const float2 (&v)[NPR]) {
  if constexpr (NPR == 1) {
    if (n0 < N) *reinterpret_cast<float2*>(row + n0) = v[0];
  } else {
#pragma unroll
    for (int k = 0; k < NPR / 2; ++k)
      if (n0 + 4 * k < N)
        *reinterpret_cast<float4*>(row + n0 + 4 * k) =
            make_float4(v[2 * k].x, v[2 * k].y, v[2 * k + 1].x, v[2 * k + 1].y);
  }
}
template <int NPR>
__device__ __forceinline__ void ld_pairs_row(const float* row, int n0, int N, float2 (&out)[NPR]) {
  if constexpr (NPR == 1) {
    out[0] = n0 < N ? *reinterpret_cast<const float2*>(row + n0) : make_float2(0.f, 0.f);
  } else {
#pragma unroll
    for (int k = 0; k < NPR / 2; ++k) {
      const float4 v = n0 + 4 * k < N ? *reinterpret_cast<const float4*>(row + n0 + 4 * k)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
      out[2 * k] = make_float2(v.x, v.y);
      out[2 * k + 1] = make_float2(v.z, v.w);
    }
  }
}
template <int NPR>
__device__ __forceinline__ void ld_pairs(const float* p, float2 (&out)[NPR]) {
  if constexpr (NPR == 1) {
    out[0] = *reinterpret_cast<const float2*>(p);
  } else {
#pragma unroll
    for (int k = 0; k < NPR / 2; ++k) {
      const float4 v = *reinterpret_cast<const float4*>(p + 4 * k);
      out[2 * k] = make_float2(v.x, v.y);
      out[2 * k + 1] = make_float2(v.z, v.w);
    }
  }
}

// ---- asynchronous global->shared copies (cp.async, completion tracked by commit groups) ----
// A source size of 0 writes zeros: that is how rows past T and channels past d_inner stay 0.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_addr(dst)),
               "l"(src), "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_addr(dst)), "l"(src),
               "r"(valid ? 4 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Stages rows t0 .. t0+kChunk-1 of a row-major [.., T, W] tensor, columns col0 .. col0+TW-1,
// into a [kChunk][TW] shared tile with cp.async; rows past T and columns past W become zeros.
// VEC needs W % 4 == 0 and col0 % 4 == 0 (then every 16-byte piece is inside or outside W).
// len: elements of src (the bounds-checked build checks every copy against it).
template <int TW, int NTH, bool VEC>
__device__ __forceinline__ void stage_tile(float* dst, const float* src, size_t row0, int t0,
                                           int T, int W, int col0, size_t len) {
  if constexpr (VEC) {
    for (int q = threadIdx.x; q < kChunk * TW / 4; q += NTH) {
      const int i = q / (TW / 4), col = (q % (TW / 4)) * 4;
      const size_t off = (row0 + t0 + i) * W + col0 + col;
      const bool v = (t0 + i < T) && (col0 + col < W) && inb(off, 4, len);
      cp_async16(dst + i * TW + col, v ? src + off : src, v);
    }
  } else {
    for (int q = threadIdx.x; q < kChunk * TW; q += NTH) {
      const int i = q / TW, col = q % TW;
      const size_t off = (row0 + t0 + i) * W + col0 + col;
      const bool v = (t0 + i < T) && (col0 + col < W) && inb(off, 1, len);
      cp_async4(dst + i * TW + col, v ? src + off : src, v);
    }
  }
}

// ---- butterfly reduce-scatter across lanes -------------------------------------------------
// Sums v[] over the lanes that differ in the lane bits MASK, MASK/2, ..., MLO (powers of two).
// While more than one value is left, each level keeps half of them: the upper half on lanes
// whose bit is set, the lower half otherwise. Once a single value is left, the remaining
// levels are plain all-reduce steps. Afterwards v[0 .. kept) holds sums of the original
// indices rs_base(lane) + r.
template <int S, int MASK, int MLO>
struct ReduceScatter {
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (MASK >= MLO && MASK >= 1) {
      if constexpr (S >= 2) {
        constexpr int H = S / 2;
        const bool up = (lane & MASK) != 0;
#pragma unroll
        for (int i = 0; i < H; ++i) {
          const float send = up ? v[i] : v[i + H];
          const float keep = up ? v[i + H] : v[i];
          v[i] = keep + __shfl_xor_sync(kFull, send, MASK);
        }
        ReduceScatter<H, MASK / 2, MLO>::run(v, lane);
      } else {
        v[0] += __shfl_xor_sync(kFull, v[0], MASK);
        ReduceScatter<1, MASK / 2, MLO>::run(v, lane);
      }
    }
  }
  // number of values left per lane
  static __host__ __device__ constexpr int kept() {
    int s = S;
    for (int m = MASK; m >= MLO && m >= 1; m /= 2)
      if (s >= 2) s /= 2;
    return s;
  }
  // original index of v[0] on this lane
  static __device__ __forceinline__ int base(int lane) {
    int b = 0, s = S;
#pragma unroll
    for (int m = MASK; m >= MLO && m >= 1; m /= 2) {
      if (s >= 2) {
        s /= 2;
        if (lane & m) b += s;
      }
    }
    return b;
  }
  // true on one lane of each group that the all-reduce levels left with equal values
  static __device__ __forceinline__ bool writer(int lane) {
    int s = S;
    bool w = true;
#pragma unroll
    for (int m = MASK; m >= MLO && m >= 1; m /= 2) {
      if (s >= 2) s /= 2;
      else if (lane & m) w = false;
    }
    return w;
  }
};

}  // namespace mscan

namespace mscan {

// ---- tensor memory (tcgen05, sm_100 family) -------------------------------------------------
// A CTA allocates columns of the SM's 128-lane x 512-column tensor memory; warp w of the CTA
// reaches lanes 32*(w%4) .. 32*(w%4)+31, and with the 32x32b shape each thread reads and writes
// its own lane. Allocation blocks while the SM has too few free columns, so a kernel must cap
// its resident CTAs per SM (through its shared memory) at 512 / columns.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {   // one warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_addr(slot)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // one warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 16 consecutive 32-bit columns of the thread's lane, from / to 8 float2 registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float2 (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "f"(v[0].x), "f"(v[0].y), "f"(v[1].x), "f"(v[1].y), "f"(v[2].x), "f"(v[2].y), "f"(v[3].x),
      "f"(v[3].y), "f"(v[4].x), "f"(v[4].y), "f"(v[5].x), "f"(v[5].y), "f"(v[6].x), "f"(v[6].y),
      "f"(v[7].x), "f"(v[7].y));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float2 (&v)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=f"(v[0].x), "=f"(v[0].y), "=f"(v[1].x), "=f"(v[1].y), "=f"(v[2].x), "=f"(v[2].y),
        "=f"(v[3].x), "=f"(v[3].y), "=f"(v[4].x), "=f"(v[4].y), "=f"(v[5].x), "=f"(v[5].y),
        "=f"(v[6].x), "=f"(v[6].y), "=f"(v[7].x), "=f"(v[7].y)
      : "r"(taddr));
}
// Completion of the thread's earlier tcgen05.st (before reading the columns back).
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Completion of tcgen05.ld into v. The registers are in-out operands so that no use of them
// is scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(float2 (&v)[8]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+f"(v[0].x), "+f"(v[0].y), "+f"(v[1].x), "+f"(v[1].y), "+f"(v[2].x),
                 "+f"(v[2].y), "+f"(v[3].x), "+f"(v[3].y), "+f"(v[4].x), "+f"(v[4].y),
                 "+f"(v[5].x), "+f"(v[5].y), "+f"(v[6].x), "+f"(v[6].y), "+f"(v[7].x),
                 "+f"(v[7].y));
}

}  // namespace mscan

namespace mscan {

// ---- mbarrier + TMA (cp.async.bulk.tensor) --------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
// Makes barrier initialisation and earlier generic-proxy shared-memory writes visible to the
// async proxy (the TMA unit) before it touches that memory.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Waits for the barrier phase with the given parity, for limit_ns at most (one second unless a
// caller asks for less). Returns false when the wait gave up (the caller records the fault;
// the kernel still runs to its end).
constexpr uint64_t kWaitLimitNs = 1000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int k = 0; k < 64; ++k)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}
// Tiled TMA loads global -> shared; completion is counted on the barrier in bytes. Elements
// outside the tensor arrive as zeros.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
      "l"(map), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_addr(dst)),
      "l"(map), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
// 16-byte predicated store without a branch.
__device__ __forceinline__ void st_global4_if(float* p, float4 v, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %5, 0;\n\t@q st.global.v4.f32 [%0], {%1, %2, %3, %4};\n\t}"
      ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"((unsigned)pred) : "memory");
}

// ---- bf16 I/O --------------------------------------------------------------------------------
// bf16 tensors are passed as raw 16-bit patterns. Widening to fp32 is exact (the bf16 bits are
// the upper half of the fp32 word); narrowing rounds to nearest even (cvt.rn).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;   // the first source goes to the upper half
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// st.global of one bf16 when a < b (as st_global_lt)
__device__ __forceinline__ void st_global_bf16_lt(uint16_t* p, float v, int a, int b) {
  asm volatile(
      "{\n\t.reg .pred q;\n\t.reg .b16 h;\n\tsetp.lt.s32 q, %2, %3;\n\t"
      "cvt.rn.bf16.f32 h, %1;\n\t@q st.global.b16 [%0], h;\n\t}"
      ::"l"(p), "f"(v), "r"(a), "r"(b) : "memory");
}
// four consecutive bf16 (8-byte aligned) when pred
__device__ __forceinline__ void st_global_bf16x4_if(uint16_t* p, float4 v, bool pred) {
  const uint32_t lo = pack_bf16x2(v.x, v.y), hi = pack_bf16x2(v.z, v.w);
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %3, 0;\n\t@q st.global.v2.b32 [%0], {%1, %2};\n\t}"
      ::"l"(p), "r"(lo), "r"(hi), "r"((unsigned)pred) : "memory");
}

// cp.async of a [kChunk][TW] bf16 tile (rows t0.., columns col0..; zeros past T or W) into the
// first half of the fp32 slot dst, 8 elements per copy (TW and W multiples of 8).
template <int TW, int NTH>
__device__ __forceinline__ void stage_tile_bf16(float* dst, const uint16_t* src, size_t row0,
                                                int t0, int T, int W, int col0, size_t len) {
  static_assert(TW % 8 == 0, "bf16 tiles move in 16-byte groups");
  uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
  for (int q = threadIdx.x; q < kChunk * TW / 8; q += NTH) {
    const int i = q / (TW / 8), col = (q % (TW / 8)) * 8;
    const size_t off = (row0 + t0 + i) * W + col0 + col;
    const bool v = (t0 + i < T) && (col0 + col < W) && inb(off, 8, len);
    cp_async16(d16 + i * TW + col, v ? src + off : src, v);
  }
}

// Widens a bf16 tile of E elements to fp32. read() takes this thread's 16-byte groups into
// registers and write() stores them widened. In place (the bf16 tile in the first half of its
// own fp32 slot) a barrier must separate the two, since the fp32 writes cover groups that other
// threads read; into another slot none is needed.
template <int E, int NTH>
struct BfTile {
  static_assert(E % 8 == 0, "whole 16-byte groups");
  static constexpr int kGroups = E / 8;
  static constexpr int kPer = (kGroups + NTH - 1) / NTH;
  uint4 r[kPer];
  __device__ __forceinline__ void read(const float* slot) {
    const uint4* s = reinterpret_cast<const uint4*>(slot);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int g = threadIdx.x + j * NTH;
      if (kGroups % NTH == 0 || g < kGroups) r[j] = s[g];
    }
  }
  __device__ __forceinline__ void write(float* slot) const {
    float4* d = reinterpret_cast<float4*>(slot);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int g = threadIdx.x + j * NTH;
      if (kGroups % NTH == 0 || g < kGroups) {
        d[2 * g] = make_float4(bf16_lo(r[j].x), bf16_hi(r[j].x), bf16_lo(r[j].y), bf16_hi(r[j].y));
        d[2 * g + 1] =
            make_float4(bf16_lo(r[j].z), bf16_hi(r[j].z), bf16_lo(r[j].w), bf16_hi(r[j].w));
      }
    }
  }
};

// ---- programmatic dependent launch ---------------------------------------------------------
// The scan kernels are launched with programmatic stream serialization, so the next one can be
// scheduled while its predecessor in the stream still runs. Each of them calls pdl_wait() before
// it touches global memory: that returns once the preceding kernel has completed and its writes
// are visible (at once when there is no such kernel). The forward and the tensor-memory
// backward call pdl_release() right after. The next kernel may then launch once every CTA of
// the grid has started (its last wave is resident), and its CTAs take the SM room that wave
// leaves as it finishes. A launch without the attribute makes both no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_release() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

}  // namespace mscan
