// fp8 (E4M3) KV blocks: the quantising KV write and decode attention over
// an fp8 pool.
//
// "PagedAttention 核心创新深度分析" §3.5 gives each attention layer's KV spec a
// quantisation mode, and its outlook (§7) names quantisation-aware blocks; the
// pages fix no format. This library stores OCP E4M3 codes with one fp32 scale
// per pool (K and V): code = e4m3(x / scale), rounded to nearest even and
// saturated to +-448 by the hardware conversion; value = code * scale. The
// pool layout is the 16-bit one with 1-byte elements, so a slot, a block and
// the block table mean the same thing; half the bytes per token are read.
//
// Attention over fp8 pools runs on the tensor-core kernel of decode_mma.cu
// for 16-bit queries, head size 128 and blocks of at least 8 tokens (any
// group size); the kernel here covers the rest (fp32 queries, head size 64,
// smaller blocks) on the CUDA cores: lane groups own token rows (8 codes per
// lane, 8-byte loads), scores and the softmax as in decode_simt.cu; k_scale is
// folded into q and v_scale into the result, so codes are only widened.
#include <cuda_fp8.h>

#include "common.cuh"
#include "launchers.h"
#include "mma_util.cuh"

namespace pa {

template <typename T> struct Wide;   // 8 stored input elements -> 8 floats
template <> struct Wide<float> {
  __device__ __forceinline__ static void load8(const float* p, float* f) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
};
template <> struct Wide<__half> {
  __device__ __forceinline__ static void load8(const __half* p, float* f) {
    Vec<__half>::to_f32(*reinterpret_cast<const uint4*>(p), f);
  }
};
template <> struct Wide<__nv_bfloat16> {
  __device__ __forceinline__ static void load8(const __nv_bfloat16* p, float* f) {
    Vec<__nv_bfloat16>::to_f32(*reinterpret_cast<const uint4*>(p), f);
  }
};

// 8 codes (one 64-bit word) -> 8 floats, exactly.
__device__ __forceinline__ void e4m3x8_to_f32(uint2 u, float* f) {
  const uint32_t w[2] = {u.x, u.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t h[2];
    e4m3x4_to_f16x2x2(w[i], h[0], h[1]);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&h[j]));
      f[4 * i + 2 * j] = v.x;
      f[4 * i + 2 * j + 1] = v.y;
    }
  }
}

// One thread per 8 elements of a (token, kv head) row, K and V together:
// widen, divide by the pool's scale (IEEE fp32), convert to E4M3 (nearest
// even, saturating), store 8 bytes at the slot's row.
template <typename T>
__global__ void reshape_and_cache_fp8_kernel(const T* __restrict__ k, const T* __restrict__ v,
                                             int64_t num_tokens, int num_kv_heads, int D,
                                             const int64_t* __restrict__ slots,
                                             uint8_t* __restrict__ kc, uint8_t* __restrict__ vc,
                                             int64_t num_blocks, int block_size, float k_scale,
                                             float v_scale, int* err) {
  const int per_row = D / 8;
  const int64_t n = num_tokens * num_kv_heads * per_row;
  const int64_t limit = num_blocks * block_size;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t c = i % per_row;
    const int64_t th = i / per_row;
    const int64_t h = th % num_kv_heads;
    const int64_t t = th / num_kv_heads;
    const int64_t slot = slots[t];
    if (slot < 0) continue;
    if (slot >= limit) {
      if (c == 0 && h == 0) latch(err, PA_ERR_OUT_OF_RANGE);
      continue;
    }
    const int64_t blk = slot / block_size;
    const int64_t row = slot - blk * block_size;
    const int64_t src = (t * num_kv_heads + h) * D + c * 8;
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + row) * D + c * 8;
    float fk[8], fv[8];
    Wide<T>::load8(k + src, fk);
    Wide<T>::load8(v + src, fv);
    uint32_t wk[2], wv[2];
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      uint32_t ak = 0, av = 0;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int e = 4 * w + 2 * j;
        const __nv_fp8x2_storage_t pk = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(fk[e], k_scale), __fdiv_rn(fk[e + 1], k_scale)),
            __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t pv = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(fv[e], v_scale), __fdiv_rn(fv[e + 1], v_scale)),
            __NV_SATFINITE, __NV_E4M3);
        ak |= (uint32_t)pk << (16 * j);
        av |= (uint32_t)pv << (16 * j);
      }
      wk[w] = ak;
      wv[w] = av;
    }
    *reinterpret_cast<uint2*>(kc + dst) = make_uint2(wk[0], wk[1]);
    *reinterpret_cast<uint2*>(vc + dst) = make_uint2(wv[0], wv[1]);
  }
}

cudaError_t launch_reshape_and_cache_fp8(const void* k, const void* v, int64_t num_tokens,
                                         int num_kv_heads, int head_size, int dtype,
                                         const int64_t* slots, void* kc, void* vc,
                                         int64_t num_blocks, int block_size, float k_scale,
                                         float v_scale, int sm_count, cudaStream_t st, int* err) {
  if (num_tokens == 0) return cudaSuccess;
  const int64_t n = num_tokens * num_kv_heads * (head_size / 8);
  const int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  if (blocks > (int64_t)sm_count * 16) blocks = (int64_t)sm_count * 16;
#define PA_FP8_WRITE(TT)                                                                 \
  reshape_and_cache_fp8_kernel<TT><<<(unsigned)blocks, threads, 0, st>>>(                \
      (const TT*)k, (const TT*)v, num_tokens, num_kv_heads, head_size, slots, (uint8_t*)kc, \
      (uint8_t*)vc, num_blocks, block_size, k_scale, v_scale, err)
  switch (dtype) {
    case PA_F32: PA_FP8_WRITE(float); break;
    case PA_F16: PA_FP8_WRITE(__half); break;
    case PA_BF16: PA_FP8_WRITE(__nv_bfloat16); break;
    default: return cudaErrorInvalidValue;
  }
#undef PA_FP8_WRITE
  return cudaGetLastError();
}

#define kNegInf8 (-__int_as_float(0x7f800000))
constexpr int kFp8Warps = 4;

// One CTA per (partition, kv head, sequence); lane groups of D/8 lanes own a
// token row, 8 codes (8 bytes) per lane; the G query heads of the group share
// each row read. Same online softmax and merges as decode_simt.cu.
template <typename T, int D, int G, int U>
__global__ void __launch_bounds__(kFp8Warps * 32)
decode_fp8_kernel(const DecodeArgs a, float k_scale, float v_scale) {
  constexpr int TPT = D / 8;
  constexpr int TPW = 32 / TPT;
  constexpr int NW = kFp8Warps;
  const int s = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / TPT, sub = lane % TPT;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;
  const int L = a.seq_lens[s];
  T* out = reinterpret_cast<T*>(a.out);
  if (L < 0 || L > a.max_seq_len || (int64_t)L > a.table_stride * a.block_size || L == 0) {
    if (split == 0) {
      if (L != 0 && threadIdx.x == 0) latch(a.err, PA_ERR_OUT_OF_RANGE);
      for (int i = threadIdx.x; i < G * D; i += blockDim.x)
        out[((int64_t)s * Hq + (int64_t)kvh * G) * D + i] = Vec<T>::cvt_out(0.f);
    }
    return;
  }
  const int lo = window_lo(L, a.window);
  const int t0 = window_base(lo) + split * a.partition;
  if (t0 >= L) return;
  const int t1 = min(L, t0 + a.partition);
  const int nsplit = (L - window_base(lo) + a.partition - 1) / a.partition;

  float qf[G][8];
  {
    const T* qp = reinterpret_cast<const T*>(a.q) + ((int64_t)s * Hq + (int64_t)kvh * G) * D +
                  sub * 8;
    const float qs = a.scale * kLog2e * k_scale;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      Wide<T>::load8(qp + (int64_t)g * D, qf[g]);
#pragma unroll
      for (int i = 0; i < 8; ++i) qf[g][i] *= qs;
    }
  }
  const int B = a.block_size;
  const int bshift = __ffs(B) - 1;
  const int32_t* trow = a.tables + (int64_t)s * a.table_stride;
  const uint8_t* kb = reinterpret_cast<const uint8_t*>(a.kc);
  const uint8_t* vb = reinterpret_cast<const uint8_t*>(a.vc);
  float m[G], l[G], acc[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = kNegInf8; l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[g][i] = 0.f;
  }
  for (int base = t0 + warp * (U * TPW); base < t1; base += NW * U * TPW) {
    uint2 ku[U], vu[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = base + u * TPW + grp;
      ok[u] = false;
      ku[u] = make_uint2(0, 0);
      vu[u] = ku[u];
      if (t >= lo && t < t1) {
        const int64_t blk = trow[t >> bshift];
        if (blk >= 0 && blk < a.num_blocks) {
          const int64_t off = ((blk * Hkv + kvh) * B + (t & (B - 1))) * D + sub * 8;
          ku[u] = __ldg(reinterpret_cast<const uint2*>(kb + off));
          vu[u] = __ldg(reinterpret_cast<const uint2*>(vb + off));
          ok[u] = true;
        } else if (sub == 0) {
          latch(a.err, PA_ERR_OUT_OF_RANGE);
        }
      }
    }
    float x[U][G];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float kf[8];
      e4m3x8_to_f32(ku[u], kf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float d = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) d = fmaf(qf[g][i], kf[i], d);
#pragma unroll
        for (int o = TPT / 2; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        x[u][g] = ok[u] ? d : kNegInf8;
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mx = m[g];
#pragma unroll
      for (int u = 0; u < U; ++u) mx = fmaxf(mx, x[u][g]);
      if (mx == kNegInf8) continue;
      const float cc = exp2f(m[g] - mx);
      l[g] *= cc;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[g][i] *= cc;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float p = exp2f(x[u][g] - mx);
        float vf[8];
        e4m3x8_to_f32(vu[u], vf);
        l[g] += p;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[g][i] = fmaf(p, vf[i], acc[g][i]);
      }
      m[g] = mx;
    }
  }
#pragma unroll
  for (int o = TPT; o < 32; o <<= 1) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[g], o);
      const float lo = __shfl_xor_sync(0xffffffffu, l[g], o);
      const float M = fmaxf(m[g], mo);
      const float ca = (m[g] == kNegInf8) ? 0.f : exp2f(m[g] - M);
      const float cb = (mo == kNegInf8) ? 0.f : exp2f(mo - M);
      l[g] = l[g] * ca + lo * cb;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float ao = __shfl_xor_sync(0xffffffffu, acc[g][i], o);
        acc[g][i] = acc[g][i] * ca + ao * cb;
      }
      m[g] = M;
    }
  }
  __shared__ float sm_acc[NW][G][D];
  __shared__ float sm_m[NW][G], sm_l[NW][G];
  if (grp == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int i = 0; i < 8; ++i) sm_acc[warp][g][sub * 8 + i] = acc[g][i];
      if (sub == 0) { sm_m[warp][g] = m[g]; sm_l[warp][g] = l[g]; }
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
    const int g = idx / D, d = idx - g * D;
    float M = kNegInf8;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w][g]);
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = sm_m[w][g];
      const float wt = (mw == kNegInf8) ? 0.f : exp2f(mw - M);
      Ls += sm_l[w][g] * wt;
      O += sm_acc[w][g][d] * wt;
    }
    O *= v_scale;
    const int h = kvh * G + g;
    if (nsplit == 1) {
      out[((int64_t)s * Hq + h) * D + d] = Vec<T>::cvt_out(Ls > 0.f ? O / Ls : 0.f);
    } else {
      const int64_t slot = ((int64_t)s * Hq + h) * a.num_splits + split;
      a.ws_acc[slot * D + d] = O;
      if (d == 0) { a.ws_ml[2 * slot] = M; a.ws_ml[2 * slot + 1] = Ls; }
    }
  }
}

template <typename T, int D, int G>
cudaError_t launch_fp8_tdg(const DecodeArgs& a, float ks, float vs, cudaStream_t st) {
  constexpr int U = (G <= 2) ? 4 : (G == 4 ? 2 : 1);
  dim3 grid(a.num_splits, a.num_kv_heads, a.num_seqs);
  decode_fp8_kernel<T, D, G, U><<<grid, kFp8Warps * 32, 0, st>>>(a, ks, vs);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_combine(a, st);
}

template <typename T, int D>
cudaError_t launch_fp8_td(const DecodeArgs& a, float ks, float vs, cudaStream_t st) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_fp8_tdg<T, D, 1>(a, ks, vs, st);
    case 2: return launch_fp8_tdg<T, D, 2>(a, ks, vs, st);
    case 4: return launch_fp8_tdg<T, D, 4>(a, ks, vs, st);
    case 8: return launch_fp8_tdg<T, D, 8>(a, ks, vs, st);
  }
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_fp8_t(const DecodeArgs& a, float ks, float vs, cudaStream_t st) {
  if (a.head_size == 64) return launch_fp8_td<T, 64>(a, ks, vs, st);
  if (a.head_size == 128) return launch_fp8_td<T, 128>(a, ks, vs, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_fp8(const DecodeArgs& a, float k_scale, float v_scale,
                              cudaStream_t st) {
  // 16-bit queries in groups of 1, 2, 4 or 8 with head size 128 and blocks
  // of at least 8 tokens: the tensor-core kernel; everything else stays on
  // the CUDA cores
  if (mma_fp8_path_applies(a))
    return launch_decode_mma_fp8(a, k_scale, v_scale, st);
  switch (a.dtype) {
    case PA_F32: return launch_fp8_t<float>(a, k_scale, v_scale, st);
    case PA_F16: return launch_fp8_t<__half>(a, k_scale, v_scale, st);
    case PA_BF16: return launch_fp8_t<__nv_bfloat16>(a, k_scale, v_scale, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
