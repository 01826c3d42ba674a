// Shared device helpers for the paged-KV kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/pagedattn.h"

namespace pa {

// Latch the first error code seen on the device; later ones are dropped.
__device__ __forceinline__ void latch(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

// Sliding-window decode: a query attends tokens lo .. L-1 with
// lo = L - window when 0 < window < L, else 0 (window 0 = whole sequence).
// Partition 0 starts at lo rounded down to a 64-token tile, so every tile
// and TMA piece keeps the alignment of the unwindowed kernels; rows before
// lo are masked, and pieces entirely before lo are neither looked up in the
// block table nor loaded.
__device__ __forceinline__ int window_lo(int L, int window) {
  return (window > 0 && L > window) ? L - window : 0;
}
__device__ __forceinline__ int window_base(int lo) { return lo & ~63; }

// ---- 16-byte vector <-> fp32 conversion per storage type ------------------
template <typename T> struct Vec;

template <> struct Vec<float> {
  static constexpr int N = 4;  // elements per 16 bytes
  __device__ __forceinline__ static void to_f32(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  __device__ __forceinline__ static float cvt_out(float x) { return x; }
};

template <> struct Vec<__half> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void to_f32(const uint4& u, float* f) {
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __half22float2(h[i]);
      f[2 * i] = t.x; f[2 * i + 1] = t.y;
    }
  }
  __device__ __forceinline__ static __half cvt_out(float x) { return __float2half_rn(x); }
};

template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void to_f32(const uint4& u, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x; f[2 * i + 1] = t.y;
    }
  }
  __device__ __forceinline__ static __nv_bfloat16 cvt_out(float x) { return __float2bfloat16_rn(x); }
};

// Streaming 16-byte load: KV rows are read once per launch, so keep them out
// of L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

constexpr float kLog2e = 1.4426950408889634f;

// Programmatic dependent launch. The decode step's kernels are launched with
// launch_pdl, so a kernel's CTAs may start while the kernel before it in the
// stream drains: each calls griddep_wait() before its first access to
// global memory (it returns once the previous kernel has completed and its
// writes are visible, at once for a plain launch), and griddep_launch()
// early, which lets the next kernel start. Only shared-memory set-up runs
// before the wait.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace pa
