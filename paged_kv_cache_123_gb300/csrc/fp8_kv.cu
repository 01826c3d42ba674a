// fp8 (E4M3) KV blocks: the quantising KV write and decode attention over
// an fp8 pool.
//
// "PagedAttention 核心创新深度分析" §3.5 gives each attention layer's KV spec a
// quantisation mode, and its outlook (§7.4) names compression-aware blocks;
// the pages fix no format. This library stores OCP E4M3 codes, code =
// e4m3(x / scale) rounded to nearest even and saturated to +-448 by the
// hardware conversion, value = code * scale, with either one fp32 scale per
// pool (K and V), or one power-of-two scale per (block, KV head) that the
// write storing a block's first row fixes from the largest magnitude of the
// tokens it puts there (two passes: fix_block_scales_kernel, then the
// quantising write). The pool layout is the 16-bit one with 1-byte elements,
// so a slot, a block and the block table mean the same thing; half the bytes
// per token are read.
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

// Power-of-two scale of a block whose first tokens' largest magnitude is
// amax: 2^k with k = ceil(log2(amax)) - 7 kept in [-126, 127], so amax lands
// in (64, 128]; 1 for amax = 0, 2^127 for an infinite amax. Integer work on
// the fp32 encoding: the biased exponent gives floor(log2), and a nonzero
// mantissa moves it up by one.
__device__ __forceinline__ float block_scale_of(float amax) {
  if (amax == 0.f) return 1.f;
  const uint32_t b = __float_as_uint(amax);
  const int ef = (int)(b >> 23);
  int k;
  if (ef == 0) {
    k = -126;                                   // below 2^-126: clamped
  } else if (ef == 255) {
    k = 127;
  } else {
    const int c = (ef - 127) + ((b & 0x7fffffu) != 0u);
    k = min(max(c - 7, -126), 127);
  }
  return __uint_as_float((uint32_t)(k + 127) << 23);
}

// First pass of the block-scaled KV write: one warp per (token, KV head)
// whose slot is row 0 of its block. The run is that token and the tokens
// right after it in the call whose slots continue it inside the block (at
// most block_size); the largest |value| over the run fixes the block's K
// (and separately V) scale. NaN values are left out of the maximum (fmaxf
// keeps the other operand), and slots past the pool are left to the second
// pass, which skips and reports them.
template <typename T>
__global__ void fix_block_scales_kernel(const T* __restrict__ k, const T* __restrict__ v,
                                        int64_t num_tokens, int num_kv_heads, int D,
                                        const int64_t* __restrict__ slots, int64_t num_blocks,
                                        int block_size, float* __restrict__ k_scales,
                                        float* __restrict__ v_scales) {
  griddep_launch();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t limit = num_blocks * block_size;
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       w < num_tokens * num_kv_heads; w += warps) {
    const int64_t t = w / num_kv_heads;
    const int h = (int)(w - t * num_kv_heads);
    const int64_t s0 = slots[t];
    if (s0 < 0 || s0 >= limit || s0 % block_size != 0) continue;
    int n = 1;
    while (n < block_size && t + n < num_tokens && slots[t + n] == s0 + n) ++n;
    float ka = 0.f, va = 0.f;
    for (int64_t e = lane; e < (int64_t)n * D; e += 32) {
      const int64_t r = e / D;
      const int64_t off = ((t + r) * num_kv_heads + h) * D + (e - r * D);
      ka = fmaxf(ka, fabsf(static_cast<float>(k[off])));
      va = fmaxf(va, fabsf(static_cast<float>(v[off])));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      ka = fmaxf(ka, __shfl_xor_sync(0xffffffffu, ka, o));
      va = fmaxf(va, __shfl_xor_sync(0xffffffffu, va, o));
    }
    if (lane == 0) {
      const int64_t idx = (s0 / block_size) * num_kv_heads + h;
      k_scales[idx] = block_scale_of(ka);
      v_scales[idx] = block_scale_of(va);
    }
  }
}

// One thread per 8 elements of a (token, kv head) row, K and V together:
// widen, divide by the scale (IEEE fp32), convert to E4M3 (nearest even,
// saturating), store 8 bytes at the slot's row. The scale is the pool's
// (k_scale, v_scale), or, when k_scales is given, the block's entry of
// k_scales / v_scales [num_blocks][num_kv_heads].
template <typename T>
__global__ void reshape_and_cache_fp8_kernel(const T* __restrict__ k, const T* __restrict__ v,
                                             int64_t num_tokens, int num_kv_heads, int D,
                                             const int64_t* __restrict__ slots,
                                             uint8_t* __restrict__ kc, uint8_t* __restrict__ vc,
                                             int64_t num_blocks, int block_size, float k_scale,
                                             float v_scale, const float* __restrict__ k_scales,
                                             const float* __restrict__ v_scales, int* err) {
  griddep_launch();
  griddep_wait();
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
    float ksc = k_scale, vsc = v_scale;
    if (k_scales != nullptr) {
      ksc = k_scales[blk * num_kv_heads + h];
      vsc = v_scales[blk * num_kv_heads + h];
    }
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
            make_float2(__fdiv_rn(fk[e], ksc), __fdiv_rn(fk[e + 1], ksc)),
            __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t pv = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(fv[e], vsc), __fdiv_rn(fv[e + 1], vsc)),
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
                                         float v_scale, float* k_scales, float* v_scales,
                                         int sm_count, cudaStream_t st, int* err) {
  if (num_tokens == 0) return cudaSuccess;
  const int threads = 256;
  if (k_scales != nullptr) {
    // pass 1: the scales of the blocks whose first row this call writes
    const int64_t warps = num_tokens * num_kv_heads;
    int64_t blocks = (warps + threads / 32 - 1) / (threads / 32);
    if (blocks > (int64_t)sm_count * 16) blocks = (int64_t)sm_count * 16;
#define PA_FIX_SCALES(TT)                                                                  \
  launch_pdl(fix_block_scales_kernel<TT>, dim3((unsigned)blocks), dim3(threads), 0, st,    \
             (const TT*)k, (const TT*)v, num_tokens, num_kv_heads, head_size, slots,       \
             num_blocks, block_size, k_scales, v_scales)
    cudaError_t e;
    switch (dtype) {
      case PA_F32: e = PA_FIX_SCALES(float); break;
      case PA_F16: e = PA_FIX_SCALES(__half); break;
      case PA_BF16: e = PA_FIX_SCALES(__nv_bfloat16); break;
      default: return cudaErrorInvalidValue;
    }
#undef PA_FIX_SCALES
    if (e != cudaSuccess) return e;
  }
  const int64_t n = num_tokens * num_kv_heads * (head_size / 8);
  int64_t blocks = (n + threads - 1) / threads;
  if (blocks > (int64_t)sm_count * 16) blocks = (int64_t)sm_count * 16;
#define PA_FP8_WRITE(TT)                                                                   \
  launch_pdl(reshape_and_cache_fp8_kernel<TT>, dim3((unsigned)blocks), dim3(threads), 0, st, \
             (const TT*)k, (const TT*)v, num_tokens, num_kv_heads, head_size, slots,         \
             (uint8_t*)kc, (uint8_t*)vc, num_blocks, block_size, k_scale, v_scale, k_scales,  \
             v_scales, err)
  switch (dtype) {
    case PA_F32: return PA_FP8_WRITE(float);
    case PA_F16: return PA_FP8_WRITE(__half);
    case PA_BF16: return PA_FP8_WRITE(__nv_bfloat16);
  }
#undef PA_FP8_WRITE
  return cudaErrorInvalidValue;
}

#define kNegInf8 (-__int_as_float(0x7f800000))
constexpr int kFp8Warps = 4;

// One CTA per (partition, kv head, sequence); lane groups of D/8 lanes own a
// token row, 8 codes (8 bytes) per lane; the G query heads of the group share
// each row read. Same online softmax and merges as decode_simt.cu. SCALED:
// the blocks carry their own scales (a.k_scales / a.v_scales), read with the
// token's codes; a token's logit is multiplied by its block's K scale and its
// softmax weight by its block's V scale before the weighted sum (the
// denominator sums the weights alone).
template <typename T, int D, int G, int U, bool SCALED>
__global__ void __launch_bounds__(kFp8Warps * 32)
decode_fp8_kernel(const DecodeArgs a, float k_scale, float v_scale) {
  constexpr int TPT = D / 8;
  constexpr int TPW = 32 / TPT;
  constexpr int NW = kFp8Warps;
  const int s = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / TPT, sub = lane % TPT;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;
  griddep_launch();
  griddep_wait();
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
    float ksu[U], vsu[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = base + u * TPW + grp;
      ok[u] = false;
      ku[u] = make_uint2(0, 0);
      vu[u] = ku[u];
      ksu[u] = vsu[u] = 1.f;
      if (t >= lo && t < t1) {
        const int64_t blk = trow[t >> bshift];
        if (blk >= 0 && blk < a.num_blocks) {
          const int64_t off = ((blk * Hkv + kvh) * B + (t & (B - 1))) * D + sub * 8;
          ku[u] = __ldg(reinterpret_cast<const uint2*>(kb + off));
          vu[u] = __ldg(reinterpret_cast<const uint2*>(vb + off));
          if (SCALED) {
            ksu[u] = __ldg(a.k_scales + blk * Hkv + kvh);
            vsu[u] = __ldg(a.v_scales + blk * Hkv + kvh);
          }
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
        x[u][g] = ok[u] ? (SCALED ? d * ksu[u] : d) : kNegInf8;
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
        const float pv = SCALED ? p * vsu[u] : p;
        float vf[8];
        e4m3x8_to_f32(vu[u], vf);
        l[g] += p;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[g][i] = fmaf(pv, vf[i], acc[g][i]);
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
  const cudaError_t e =
      a.k_scales != nullptr
          ? launch_pdl(decode_fp8_kernel<T, D, G, U, true>, grid, dim3(kFp8Warps * 32), 0, st, a,
                       1.f, 1.f)
          : launch_pdl(decode_fp8_kernel<T, D, G, U, false>, grid, dim3(kFp8Warps * 32), 0, st, a,
                       ks, vs);
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
