// Warp-level tensor-core and shared-memory helpers shared by the
// tensor-core attention kernels: mma.sync m16n8k16 for fp16/bf16 with fp32
// accumulation, ldmatrix loads, movmatrix transposes, and the address
// arithmetic of the TMA 128-byte swizzle.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

namespace pa {

template <typename T> struct MmaOps;

template <> struct MmaOps<__nv_bfloat16> {
  static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  __device__ __forceinline__ static void mma(float* c, const uint32_t* a, uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __device__ __forceinline__ static float2 unpack(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
  }
};

template <> struct MmaOps<__half> {
  static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  __device__ __forceinline__ static void mma(float* c, const uint32_t* a, uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __device__ __forceinline__ static float2 unpack(uint32_t u) {
    return __half22float2(*reinterpret_cast<__half2*>(&u));
  }
};

__device__ __forceinline__ void ldsm_x4(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Shared-memory address of 16-byte chunk `dch` (0 .. D/8-1) of token row
// `row` in a tile of whole rows stored as 128-byte lines (HALVES lines per
// row), with the TMA 128-byte swizzle: the 16-byte chunk index inside a line
// is XORed with the line index mod 8. The tile starts on a 1024-byte boundary.
template <int HALVES>
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int dch) {
  const int line = row * HALVES + (dch >> 3);
  return base + line * 128 + (((dch & 7) ^ (line & 7)) << 4);
}

// A pair of query values of type T as the operand type MT of the products.
template <typename T, typename MT>
__device__ __forceinline__ uint32_t to_mma_pair(uint32_t v) {
  if constexpr (std::is_same<T, MT>::value) {
    return v;
  } else {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
    const __half2 h = __floats2half2_rn(f.x, f.y);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

// Four E4M3 codes (one 32-bit word, lowest byte first) -> two fp16 pairs,
// exactly (every E4M3 value is an fp16 value): lo holds bytes 0 and 1 (byte 0
// in the low half), hi bytes 2 and 3. One PTX conversion per 16-bit half of
// the word, with no masking, shifting or repacking around it.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 c0, c1;\n\t"
      "mov.b32 {c0, c1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, c0;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, c1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

}  // namespace pa
