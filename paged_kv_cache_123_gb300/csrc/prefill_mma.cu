// Causal paged attention for several new tokens per sequence (chunked
// prefill, speculative tokens), on the tensor cores.
//
// "vLLM 的 PagedAttention：显存管理如何撑起大模型推理" §2.5: the scheduler
// gives each request a token budget per step, so a step may append many
// tokens to a request (a prefill chunk) or a few (speculative candidates);
// "PagedAttention 核心创新深度分析" §2.3: the slot mapping already places any
// number of tokens per request. New token i of sequence s (n_s new tokens,
// L_s tokens in the pool including them) sits at position L_s - n_s + i and
// attends to positions 0 .. L_s - n_s + i, read through the block table.
//
// This file holds the short runs — at most 16 (token, head) columns per KV
// head, e.g. one or two speculative tokens of a GQA group of 8 — on
// mma.sync in the decode kernel's layout, and the log-sum-exp combine of KV
// partitions shared with the tcgen05 kernel (prefill_tc.cu), which takes
// every longer run. K/V tiles of 64 tokens arrive by the same TMA / mbarrier
// ring as the decode kernel (one 4-D box per block, 128-byte swizzle).
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "launchers.h"
#include "mma_util.cuh"
#include "tma.cuh"

namespace pa {
namespace {

constexpr int kMqConsumers = 4;
constexpr int kMqThreads = (kMqConsumers + 1) * 32;
constexpr int kMqTile = 64;        // KV tokens per stage
constexpr int kMqStages = 3;
constexpr long long kMqWaitCycles = 4000000000LL;
#define kNegInfQ (-__int_as_float(0x7f800000))
constexpr float kLazyLog2Q = 8.f;   // reference maximum moves when exceeded by 2^8

// Producer warp: fill the ring with the KV tiles [0, ntiles) of (sequence,
// kv head): lane p issues the TMA loads (whole rows, one 4-D box per block
// piece) of the tile's block-piece p.
template <int ROW_BYTES, int KV_BYTES, int STAGE_BYTES>
__device__ void mq_produce(const MultiQueryArgs& a, const CUtensorMap* tmK,
                           const CUtensorMap* tmV, const int32_t* trow, int kvh, int kv_lo,
                           int kv_end, int ntiles, uint32_t smem0, uint32_t bar0, unsigned* tile_mask,
                           volatile int* abort_flag, int lane) {
  const int B = a.block_size;
  const int bshift = __ffs(B) - 1;
  const int R = B < kMqTile ? B : kMqTile;
  const int npieces = kMqTile / R;
  if (lane == 0) {
    prefetch_tensormap(tmK);
    prefetch_tensormap(tmV);
  }
  int issued = 0;
  for (int i = 0; i < ntiles; ++i) {
    const int st = i % kMqStages;
    const int ts = kv_lo + i * kMqTile;
    const int te = min(kv_end, ts + kMqTile);
    const int tok = ts + lane * R;
    int64_t blk = -1;
    bool mine = false;
    if (lane < npieces && tok < te) {
      blk = trow[tok >> bshift];
      mine = blk >= 0 && blk < a.num_blocks;
      if (!mine) latch(a.err, PA_ERR_OUT_OF_RANGE);
    }
    const unsigned pm = __ballot_sync(0xffffffffu, mine);
    int ok = 1;
    if (lane == 0) {
      if (i >= kMqStages)
        ok = mbar_wait_bounded(bar0 + 8u * (kMqStages + st), ((i / kMqStages) - 1) & 1,
                               abort_flag, kMqWaitCycles);
      if (ok) {
        tile_mask[st] = pm;
        mbar_arrive_expect_tx(bar0 + 8u * st, (uint32_t)__popc(pm) * 2u * R * ROW_BYTES);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) break;
    if (mine) {
      const uint32_t kdst = smem0 + st * STAGE_BYTES + lane * R * ROW_BYTES;
      const int z = (int)(blk * a.num_kv_heads + kvh);
      const int y = tok & (B - 1);
      tma_load_4d(kdst, tmK, 0, 0, y, z, bar0 + 8u * st);
      tma_load_4d(kdst + KV_BYTES, tmV, 0, 0, y, z, bar0 + 8u * st);
    }
    issued = i + 1;
  }
  // let this warp's copies land before the CTA can leave (also after a
  // timeout: this wait has its own limit and ignores the abort flag)
  if (lane == 0)
    for (int j = issued > kMqStages ? issued - kMqStages : 0; j < issued; ++j)
      mbar_wait_drain(bar0 + 8u * (j % kMqStages), (j / kMqStages) & 1, kMqWaitCycles);
}

// Log-sum-exp merge of the partitions of one (new token, query head) row;
// rows whose keys fit one partition were written by the attention kernel.
template <typename T, int D>
__global__ void __launch_bounds__(D) mq_combine_kernel(const MultiQueryArgs a) {
  const int64_t t = blockIdx.x;
  const int head = blockIdx.y, d = threadIdx.x;
  int lo = 0, hi = a.num_seqs + 1;              // owning sequence of row t
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)a.qsl[mid] <= t) lo = mid + 1; else hi = mid;
  }
  const int s = lo - 1;
  if (s < 0 || s >= a.num_seqs) return;
  const int q0 = a.qsl[s], n = a.qsl[s + 1] - q0, L = a.seq_lens[s];
  if (n < 0 || n > a.max_query_len || L < n || L > a.max_seq_len ||
      (int64_t)L > a.table_stride * a.block_size || q0 < 0)
    return;
  const int pos = L - n + (int)(t - q0);
  const int count = (pos + a.partition) / a.partition;
  if (count <= 1) return;
  const int64_t base = (t * a.num_q_heads + head) * a.num_splits;
  float M = kNegInfQ;
  for (int p = 0; p < count; ++p) M = fmaxf(M, a.ws_ml[2 * (base + p)]);
  float Ls = 0.f, O = 0.f;
  for (int p = 0; p < count; ++p) {
    const float mp = a.ws_ml[2 * (base + p)];
    const float w = (mp == kNegInfQ) ? 0.f : exp2f(mp - M);
    Ls += a.ws_ml[2 * (base + p) + 1] * w;
    O += a.ws_acc[(base + p) * D + d] * w;
  }
  T* out = reinterpret_cast<T*>(a.out);
  out[(t * a.num_q_heads + head) * D + d] = Vec<T>::cvt_out(Ls > 0.f ? O / Ls : 0.f);
}

// Few new tokens per sequence (speculative tokens): the decode kernel's
// layout. Columns are (new token, query head) pairs, query-major, 16 per CTA
// (two N = 8 tiles); each consumer warp takes 16 KV tokens of every 64-token
// tile as M, computes S^T = K Q^T and O^T += V^T P^T with mma.sync, and
// keeps a per-column softmax with that column's causal limit. The KV range
// is read once per 16 columns; the four warps merge through shared memory.
constexpr int kMqsCols = 16;

template <typename T, int D, int G>
__global__ void __launch_bounds__(kMqThreads, 2)
multi_query_cols_kernel(const MultiQueryArgs a, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV) {
  constexpr int HALVES = D / 64;
  constexpr int ROW_BYTES = HALVES * 128;
  constexpr int KV_BYTES = kMqTile * ROW_BYTES;
  constexpr int STAGE_BYTES = 2 * KV_BYTES;
  constexpr int KSTEPS = D / 16;
  constexpr int NT = kMqsCols / 8;

  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, reached by pointer arithmetic on the shared
  // array itself so the compiler keeps every access in the shared space
  // (an integer round trip would make them generic loads)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kMqStages * STAGE_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kMqStages);
  unsigned* tile_mask = reinterpret_cast<unsigned*>(bars + 2 * kMqStages) + 1;
  const uint32_t smem0 = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);

  const int s = blockIdx.z, kvh = blockIdx.y;
  const int col_tiles = (a.max_query_len * G + kMqsCols - 1) / kMqsCols;
  const int ct = blockIdx.x % col_tiles, split = blockIdx.x / col_tiles;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = a.num_q_heads;
  const int q0 = a.qsl[s];
  const int n = a.qsl[s + 1] - q0;
  const int L = a.seq_lens[s];
  if (n < 0 || n > a.max_query_len || L < n || L > a.max_seq_len ||
      (int64_t)L > a.table_stride * a.block_size || q0 < 0) {
    if (blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0) latch(a.err, PA_ERR_OUT_OF_RANGE);
    return;
  }
  const int c0 = ct * kMqsCols;
  if (c0 >= n * G) return;
  const int i_last = min(n - 1, (c0 + kMqsCols - 1) / G);
  const int kv_all = L - n + i_last + 1;
  const int kv_lo = split * a.partition;
  if (kv_lo >= kv_all) return;
  const int kv_end = min(kv_all, kv_lo + a.partition);
  const int ntiles = (kv_end - kv_lo + kMqTile - 1) / kMqTile;
  const int32_t* trow = a.tables + (int64_t)s * a.table_stride;
  const int B = a.block_size;
  const int R = B < kMqTile ? B : kMqTile;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kMqStages; ++st) {
      mbar_init(bar0 + 8u * st, 1);
      mbar_init(bar0 + 8u * (kMqStages + st), kMqConsumers);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();

  const int c = lane & 3, n8 = lane >> 2;
  float o[NT][KSTEPS][4];
  float m[NT][2], l[NT][2];
  int cpos[NT][2];        // causal limit of this lane's two columns per N tile (-1: none)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt][0] = m[nt][1] = kNegInfQ;
    l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int col = c0 + nt * 8 + 2 * c + e;
      cpos[nt][e] = (col / G < n) ? L - n + col / G : -1;
    }
  }

  if (warp == kMqConsumers) {
    mq_produce<ROW_BYTES, KV_BYTES, STAGE_BYTES>(a, &tmK, &tmV, trow, kvh, kv_lo, kv_end,
                                                        ntiles, smem0, bar0, tile_mask, abort_flag,
                                                 lane);
  } else {
    uint32_t qf[NT][KSTEPS][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int col = c0 + nt * 8 + n8;
      const bool live = col / G < n;
      const T* qb = reinterpret_cast<const T*>(a.q) +
                    ((int64_t)(q0 + (live ? col / G : 0)) * Hq + (int64_t)kvh * G + col % G) * D;
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        qf[nt][ks][0] = live ? *reinterpret_cast<const uint32_t*>(qb + ks * 16 + 2 * c) : 0u;
        qf[nt][ks][1] = live ? *reinterpret_cast<const uint32_t*>(qb + ks * 16 + 8 + 2 * c) : 0u;
      }
    }
    const float sl2 = a.scale * kLog2e;
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % kMqStages;
      if (!mbar_wait_bounded(bar0 + 8u * st, (i / kMqStages) & 1, abort_flag, kMqWaitCycles))
        break;
      const int ts = kv_lo + i * kMqTile;
      const int te = min(kv_end, ts + kMqTile);
      const int r0 = ts + warp * 16;
      const uint32_t kst = smem0 + st * STAGE_BYTES;
      const uint32_t vst = kst + KV_BYTES;
      if (r0 < te) {
        const int rr = warp * 16 + (lane & 15);
        const bool row_ok = (ts + rr < te) && ((tile_mask[st] >> (rr / R)) & 1u);
        const unsigned okm = __ballot_sync(0xffffffffu, row_ok) & 0xffffu;
        if (okm != 0xffffu) {          // clear this warp's V rows without a token
          const int r = lane & 15, h = lane >> 4;
          if (h < HALVES && !((okm >> r) & 1u)) {
            uint4* p = reinterpret_cast<uint4*>(smem + (vst - smem0) + (warp * 16 + r) * ROW_BYTES +
                                                h * 128);
#pragma unroll
            for (int j = 0; j < 8; ++j) p[j] = make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
        }
        const int jA = r0 + n8, jB = jA + 8;          // this lane's two KV tokens
        const bool okA = (okm >> n8) & 1u, okB = (okm >> (n8 + 8)) & 1u;
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float sacc[4] = {0.f, 0.f, 0.f, 0.f};
          const int jj = lane >> 3;
          const int row = warp * 16 + (jj & 1) * 8 + (lane & 7);
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            uint32_t af[4];
            ldsm_x4(af, swz<HALVES>(kst, row, ks * 2 + (jj >> 1)));
            MmaOps<T>::mma(sacc, af, qf[nt][ks][0], qf[nt][ks][1]);
          }
          float x[4];
          x[0] = (okA && jA <= cpos[nt][0]) ? sacc[0] * sl2 : kNegInfQ;
          x[1] = (okA && jA <= cpos[nt][1]) ? sacc[1] * sl2 : kNegInfQ;
          x[2] = (okB && jB <= cpos[nt][0]) ? sacc[2] * sl2 : kNegInfQ;
          x[3] = (okB && jB <= cpos[nt][1]) ? sacc[3] * sl2 : kNegInfQ;
          float mx[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], off));
            mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], off));
          }
          // lazy reference (as in the decode kernel): a column's reference
          // maximum moves to the tile's maximum only when that exceeds it
          // by more than 2^8, so the weights stay below 2^8 and the output
          // is rescaled only on those tiles, in a warp-uniform branch
          float p[4], al[2] = {1.f, 1.f};
          bool up[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) up[e] = mx[e] > m[nt][e] + kLazyLog2Q;
          const bool rescale = __any_sync(0xffffffffu, up[0] || up[1]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            if (up[e]) {
              al[e] = exp2f(m[nt][e] - mx[e]);     // 0 on the first tile
              m[nt][e] = mx[e];
            }
            const bool live = m[nt][e] != kNegInfQ;
            p[e] = live ? exp2f(x[e] - m[nt][e]) : 0.f;
            p[e + 2] = live ? exp2f(x[e + 2] - m[nt][e]) : 0.f;
          }
          const uint32_t cA = MmaOps<T>::pack(p[0], p[1]);
          const uint32_t cB = MmaOps<T>::pack(p[2], p[3]);
          const float2 fA = MmaOps<T>::unpack(cA), fB = MmaOps<T>::unpack(cB);
          l[nt][0] = l[nt][0] * al[0] + fA.x + fB.x;
          l[nt][1] = l[nt][1] * al[1] + fA.y + fB.y;
          if (rescale) {
#pragma unroll
            for (int mt = 0; mt < KSTEPS; ++mt) {
              o[nt][mt][0] *= al[0]; o[nt][mt][1] *= al[1];
              o[nt][mt][2] *= al[0]; o[nt][mt][3] *= al[1];
            }
          }
          pb[nt][0] = movmatrix_trans(cA);
          pb[nt][1] = movmatrix_trans(cB);
        }
        {
          const int jj = lane >> 3;
          const int row = warp * 16 + (jj >> 1) * 8 + (lane & 7);
#pragma unroll
          for (int mt = 0; mt < KSTEPS; ++mt) {
            uint32_t af[4];
            ldsm_x4_trans(af, swz<HALVES>(vst, row, mt * 2 + (jj & 1)));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) MmaOps<T>::mma(o[nt][mt], af, pb[nt][0], pb[nt][1]);
          }
        }
        if (okm != 0xffffu) fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar0 + 8u * (kMqStages + st));
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1)
          l[nt][e] += __shfl_xor_sync(0xffffffffu, l[nt][e], off);
  }
  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) latch(a.err, PA_ERR_TIMEOUT);
    return;
  }
  float* sm_o = reinterpret_cast<float*>(smem);            // [4][16][D]
  float* sm_m = sm_o + kMqConsumers * kMqsCols * D;          // [4][16]
  float* sm_l = sm_m + kMqConsumers * kMqsCols;              // [4][16]
  if (warp < kMqConsumers) {
    float* base = sm_o + warp * kMqsCols * D;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) {
        const int cl = nt * 8 + 2 * c, d = mt * 16 + n8;
        base[cl * D + d] = o[nt][mt][0];
        base[(cl + 1) * D + d] = o[nt][mt][1];
        base[cl * D + d + 8] = o[nt][mt][2];
        base[(cl + 1) * D + d + 8] = o[nt][mt][3];
      }
      if (n8 == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          sm_m[warp * kMqsCols + nt * 8 + 2 * c + e] = m[nt][e];
          sm_l[warp * kMqsCols + nt * 8 + 2 * c + e] = l[nt][e];
        }
      }
    }
  }
  __syncthreads();
  T* out = reinterpret_cast<T*>(a.out);
  for (int idx = threadIdx.x; idx < kMqsCols * D; idx += blockDim.x) {
    const int cl = idx / D, d = idx - cl * D;
    const int col = c0 + cl;
    const int qi = col / G;
    if (qi >= n) continue;
    float M = kNegInfQ;
#pragma unroll
    for (int w = 0; w < kMqConsumers; ++w) M = fmaxf(M, sm_m[w * kMqsCols + cl]);
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kMqConsumers; ++w) {
      const float mw = sm_m[w * kMqsCols + cl];
      const float wt = (mw == kNegInfQ) ? 0.f : exp2f(mw - M);
      Ls += sm_l[w * kMqsCols + cl] * wt;
      O += sm_o[(w * kMqsCols + cl) * D + d] * wt;
    }
    const int pos = L - n + qi;
    const int count = (pos + a.partition) / a.partition;
    const int64_t t = q0 + qi;
    const int head = kvh * G + col % G;
    if (count == 1) {
      if (split == 0)
        out[(t * Hq + head) * D + d] = Vec<T>::cvt_out(Ls > 0.f ? O / Ls : 0.f);
    } else if (split < count) {
      const int64_t slot = (t * Hq + head) * a.num_splits + split;
      a.ws_acc[slot * D + d] = O;
      if (d == 0) { a.ws_ml[2 * slot] = M; a.ws_ml[2 * slot + 1] = Ls; }
    }
  }
}

}  // namespace

namespace {

template <int D>
constexpr int mq_smem_bytes() {
  return 1024 + kMqStages * 2 * kMqTile * (D / 64) * 128 + 2 * kMqStages * 8 + 4 +
         4 * kMqStages + 16;
}

template <typename T, int D, int G>
cudaError_t launch_mq_tdg(const MultiQueryArgs& a, cudaStream_t st) {
  const int64_t rows = (int64_t)a.max_query_len * G;   // (token, head) rows per KV head
  if (rows == 0 || a.num_seqs == 0) return cudaSuccess;
  if (rows > kMqsCols) {
    // more than 16 rows per KV head (prefill chunks, and speculative runs
    // such as 4 tokens x 8 heads): the tcgen05 kernel, 128 rows per CTA;
    // even mostly empty row tiles keep it ahead of mma.sync
    cudaError_t e = launch_multi_query_tc(a, st);
    if (e != cudaSuccess) return e;
  } else {
    // a few new tokens per sequence: columns as N, KV tokens as M
    CUtensorMap tk, tv;
    if (!encode_kv_pool_map(&tk, a.kc, a.dtype, a.num_blocks, a.num_kv_heads, a.block_size,
                            a.head_size) ||
        !encode_kv_pool_map(&tv, a.vc, a.dtype, a.num_blocks, a.num_kv_heads, a.block_size,
                            a.head_size))
      return cudaErrorInvalidValue;
    constexpr int smem = mq_smem_bytes<D>();
    static std::once_flag once_cols;
    static cudaError_t attr_cols = cudaSuccess;
    std::call_once(once_cols, []() {
      attr_cols = cudaFuncSetAttribute(multi_query_cols_kernel<T, D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr_cols != cudaSuccess) return attr_cols;
    dim3 grid((unsigned)a.num_splits, a.num_kv_heads, a.num_seqs);
    multi_query_cols_kernel<T, D, G><<<grid, kMqThreads, smem, st>>>(a, tk, tv);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.num_splits <= 1) return e;
  if (a.num_tokens > 0x7fffffffLL) return cudaErrorInvalidValue;
  dim3 cgrid((unsigned)a.num_tokens, a.num_q_heads);
  mq_combine_kernel<T, D><<<cgrid, D, 0, st>>>(a);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_mq_td(const MultiQueryArgs& a, cudaStream_t st) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_mq_tdg<T, D, 1>(a, st);
    case 2: return launch_mq_tdg<T, D, 2>(a, st);
    case 4: return launch_mq_tdg<T, D, 4>(a, st);
    case 8: return launch_mq_tdg<T, D, 8>(a, st);
  }
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_mq_t(const MultiQueryArgs& a, cudaStream_t st) {
  if (a.head_size == 64) return launch_mq_td<T, 64>(a, st);
  if (a.head_size == 128) return launch_mq_td<T, 128>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_multi_query(const MultiQueryArgs& a, cudaStream_t st) {
  if (a.dtype == PA_BF16) return launch_mq_t<__nv_bfloat16>(a, st);
  if (a.dtype == PA_F16) return launch_mq_t<__half>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
