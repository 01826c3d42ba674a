// Paged decode attention on the CUDA cores, and the split-K combine.
//
// What is computed ("Visual reading: paged-attention-kv-cache", block-wise
// attention and block table section; "Infra: PagedAttention", "按 Block
// 分配"): for sequence s and query head h, with KV head kvh = h / G,
//     o = sum_j softmax_j(scale <q, k_j>) v_j ,  j < seq_lens[s]
// where k_j / v_j are row j % B of KV head kvh in physical block
// block_tables[s][j / B].
//
// Work decomposition: one CTA per (context partition, KV head, sequence).
// The partition is a run of whole blocks; a CTA serves all G query heads of
// its KV head from one read of each K/V row (GQA: the group shares the
// read). Lane groups of TPT lanes own one token row each (16 bytes per lane),
// so a warp reads TPW = 32 / TPT rows per step with coalesced 16-byte loads.
// Each lane group keeps a running (max, sum, acc) in the log2 domain and
// folds U rows per update. At the end the groups and warps are merged; a
// sequence covered by one partition writes its output directly, otherwise
// the partial (max, sum, acc) goes to the workspace and combine_kernel
// merges the partitions with log-sum-exp weights.
#include "common.cuh"
#include "launchers.h"

namespace pa {

constexpr int kSimtWarps = 4;
#define kNegInf (-__int_as_float(0x7f800000))

template <typename T, int D>
__device__ __forceinline__ void write_zero_heads(const DecodeArgs& a, int s, int h0, int G) {
  T* out = reinterpret_cast<T*>(a.out);
  for (int i = threadIdx.x; i < G * D; i += blockDim.x)
    out[((int64_t)s * a.num_q_heads + h0) * D + i] = Vec<T>::cvt_out(0.f);
}

__device__ __forceinline__ bool bad_length(const DecodeArgs& a, int L) {
  return L < 0 || L > a.max_seq_len || (int64_t)L > a.table_stride * a.block_size;
}

template <typename T, int D, int G, int U>
__global__ void __launch_bounds__(kSimtWarps * 32)
decode_simt_kernel(const DecodeArgs a) {
  constexpr int VEC = Vec<T>::N;
  constexpr int TPT = D / VEC;
  constexpr int TPW = 32 / TPT;
  constexpr int NW = kSimtWarps;
  static_assert(TPT >= 1 && TPT <= 32 && (32 % TPT) == 0, "row split");

  const int s = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / TPT, sub = lane % TPT;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;
  griddep_launch();
  griddep_wait();
  const int L = a.seq_lens[s];
  if (bad_length(a, L) || L == 0) {
    if (split == 0) {
      if (L != 0 && threadIdx.x == 0) latch(a.err, PA_ERR_OUT_OF_RANGE);
      write_zero_heads<T, D>(a, s, kvh * G, G);
    }
    return;
  }
  const int lo = window_lo(L, a.window);
  const int tb = window_base(lo);
  const int t0 = tb + split * a.partition;
  if (t0 >= L) return;
  const int t1 = min(L, t0 + a.partition);
  const int nsplit = (L - tb + a.partition - 1) / a.partition;

  // q for the G heads of this group, pre-multiplied by scale * log2(e) so
  // the softmax runs on exp2.
  float qf[G][VEC];
  {
    const T* qp = reinterpret_cast<const T*>(a.q) +
                  ((int64_t)s * Hq + (int64_t)kvh * G) * D + sub * VEC;
    const float qs = a.scale * kLog2e;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      uint4 u = *reinterpret_cast<const uint4*>(qp + (int64_t)g * D);
      Vec<T>::to_f32(u, qf[g]);
#pragma unroll
      for (int i = 0; i < VEC; ++i) qf[g][i] *= qs;
    }
  }

  const int B = a.block_size;
  const int bshift = __ffs(B) - 1;
  const int32_t* trow = a.tables + (int64_t)s * a.table_stride;
  const T* kbase = reinterpret_cast<const T*>(a.kc);
  const T* vbase = reinterpret_cast<const T*>(a.vc);

  float m[G], l[G], acc[G][VEC];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = kNegInf; l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) acc[g][i] = 0.f;
  }

  for (int base = t0 + warp * (U * TPW); base < t1; base += NW * U * TPW) {
    uint4 ku[U], vu[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = base + u * TPW + grp;
      ok[u] = false;
      ku[u] = make_uint4(0, 0, 0, 0);
      vu[u] = ku[u];
      if (t >= lo && t < t1) {
        const int64_t blk = trow[t >> bshift];
        if (blk >= 0 && blk < a.num_blocks) {
          const int64_t off = ((blk * Hkv + kvh) * B + (t & (B - 1))) * D + sub * VEC;
          ku[u] = ld_stream16(kbase + off);
          vu[u] = ld_stream16(vbase + off);
          ok[u] = true;
        } else if (sub == 0) {
          latch(a.err, PA_ERR_OUT_OF_RANGE);
        }
      }
    }
    float x[U][G];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float kf[VEC];
      Vec<T>::to_f32(ku[u], kf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float d = 0.f;
#pragma unroll
        for (int i = 0; i < VEC; ++i) d = fmaf(qf[g][i], kf[i], d);
#pragma unroll
        for (int o = TPT / 2; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        x[u][g] = ok[u] ? d : kNegInf;
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mx = m[g];
#pragma unroll
      for (int u = 0; u < U; ++u) mx = fmaxf(mx, x[u][g]);
      if (mx == kNegInf) continue;          // nothing valid yet in this group
      const float c = exp2f(m[g] - mx);     // 0 when m[g] was -inf
      l[g] *= c;
#pragma unroll
      for (int i = 0; i < VEC; ++i) acc[g][i] *= c;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float p = exp2f(x[u][g] - mx);  // 0 for invalid rows
        float vf[VEC];
        Vec<T>::to_f32(vu[u], vf);
        l[g] += p;
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc[g][i] = fmaf(p, vf[i], acc[g][i]);
      }
      m[g] = mx;
    }
  }

  // merge the TPW lane groups of the warp (lanes with equal `sub`)
#pragma unroll
  for (int o = TPT; o < 32; o <<= 1) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[g], o);
      const float lo = __shfl_xor_sync(0xffffffffu, l[g], o);
      const float M = fmaxf(m[g], mo);
      const float ca = (m[g] == kNegInf) ? 0.f : exp2f(m[g] - M);
      const float cb = (mo == kNegInf) ? 0.f : exp2f(mo - M);
      l[g] = l[g] * ca + lo * cb;
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
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
      for (int i = 0; i < VEC; ++i) sm_acc[warp][g][sub * VEC + i] = acc[g][i];
      if (sub == 0) { sm_m[warp][g] = m[g]; sm_l[warp][g] = l[g]; }
    }
  }
  __syncthreads();

  T* out = reinterpret_cast<T*>(a.out);
  for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
    const int g = idx / D, d = idx - g * D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w][g]);
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = sm_m[w][g];
      const float wt = (mw == kNegInf) ? 0.f : exp2f(mw - M);
      Ls += sm_l[w][g] * wt;
      O += sm_acc[w][g][d] * wt;
    }
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

// Log-sum-exp combine of the partitions of one (sequence, query head):
//   M = max_p m_p,  w_p = 2^(m_p - M),  o = sum_p w_p acc_p / sum_p w_p l_p
// (all in the log2 domain the partial kernel used).
template <typename T, int D>
__global__ void __launch_bounds__(D) combine_kernel(const DecodeArgs a) {
  const int s = blockIdx.y, h = blockIdx.x, d = threadIdx.x;
  griddep_launch();
  griddep_wait();
  const int L = a.seq_lens[s];
  if (bad_length(a, L) || L == 0) return;
  const int tb = window_base(window_lo(L, a.window));
  const int n = (L - tb + a.partition - 1) / a.partition;
  if (n <= 1) return;
  const int64_t base = ((int64_t)s * a.num_q_heads + h) * a.num_splits;
  // one pass, four partitions at a time (their loads issued together): the
  // running maximum M, with the sums rescaled when it grows
  float M = kNegInf, Ls = 0.f, O = 0.f;
  for (int p0 = 0; p0 < n; p0 += 4) {
    float mv[4], lv[4], av[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int p = p0 + u;
      mv[u] = kNegInf; lv[u] = 0.f; av[u] = 0.f;
      if (p < n) {
        mv[u] = a.ws_ml[2 * (base + p)];
        lv[u] = a.ws_ml[2 * (base + p) + 1];
        av[u] = a.ws_acc[(base + p) * D + d];
      }
    }
    const float Mn = fmaxf(fmaxf(M, fmaxf(mv[0], mv[1])), fmaxf(mv[2], mv[3]));
    if (Mn == kNegInf) continue;
    const float f = (M == kNegInf) ? 0.f : exp2f(M - Mn);
    Ls *= f;
    O *= f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = (mv[u] == kNegInf) ? 0.f : exp2f(mv[u] - Mn);
      Ls += lv[u] * w;
      O += av[u] * w;
    }
    M = Mn;
  }
  T* out = reinterpret_cast<T*>(a.out);
  out[((int64_t)s * a.num_q_heads + h) * D + d] = Vec<T>::cvt_out(Ls > 0.f ? O / Ls : 0.f);
}

template <typename T, int D>
cudaError_t launch_combine_td(const DecodeArgs& a, cudaStream_t st) {
  if (a.num_splits <= 1) return cudaSuccess;
  dim3 grid(a.num_q_heads, a.num_seqs);
  return launch_pdl(combine_kernel<T, D>, grid, dim3(D), 0, st, a);
}

template <typename T>
cudaError_t launch_combine_t(const DecodeArgs& a, cudaStream_t st) {
  if (a.head_size == 64) return launch_combine_td<T, 64>(a, st);
  if (a.head_size == 128) return launch_combine_td<T, 128>(a, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t st) {
  switch (a.dtype) {
    case PA_F32: return launch_combine_t<float>(a, st);
    case PA_F16: return launch_combine_t<__half>(a, st);
    case PA_BF16: return launch_combine_t<__nv_bfloat16>(a, st);
  }
  return cudaErrorInvalidValue;
}

template <typename T, int D, int G>
cudaError_t launch_simt_tg(const DecodeArgs& a, cudaStream_t st) {
  constexpr int U = (G <= 2) ? 4 : (G == 4 ? 2 : 1);
  dim3 grid(a.num_splits, a.num_kv_heads, a.num_seqs);
  const cudaError_t e = launch_pdl(decode_simt_kernel<T, D, G, U>, grid, dim3(kSimtWarps * 32),
                                   0, st, a);
  if (e != cudaSuccess) return e;
  return launch_combine_td<T, D>(a, st);
}

template <typename T, int D>
cudaError_t launch_simt_t(const DecodeArgs& a, cudaStream_t st) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_simt_tg<T, D, 1>(a, st);
    case 2: return launch_simt_tg<T, D, 2>(a, st);
    case 4: return launch_simt_tg<T, D, 4>(a, st);
    case 8: return launch_simt_tg<T, D, 8>(a, st);
  }
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_simt_d(const DecodeArgs& a, cudaStream_t st) {
  if (a.head_size == 64) return launch_simt_t<T, 64>(a, st);
  if (a.head_size == 128) return launch_simt_t<T, 128>(a, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t st) {
  switch (a.dtype) {
    case PA_F32: return launch_simt_d<float>(a, st);
    case PA_F16: return launch_simt_d<__half>(a, st);
    case PA_BF16: return launch_simt_d<__nv_bfloat16>(a, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  if (mma_path_applies(a)) return launch_decode_mma(a, st);
  return launch_decode_simt(a, st);
}

}  // namespace pa
