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
// Rows are (new token, query head) pairs of one KV head, query-major
// (row = i * G + g), so the G heads of a group share each K/V read. A CTA
// owns 64 rows; each of its four consumer warps owns 16 rows and runs the
// whole KV range up to its CTA's last position: S = Q K^T and O += P V with
// mma.sync m16n8k16 (rows as M, 8 KV tokens or 8 head dims as N), online
// softmax in the log2 domain, causal mask per row. K/V tiles of 64 tokens
// arrive by the same TMA / mbarrier ring as the decode kernel (one 4-D box per
// block, 128-byte swizzle). Tiles past every row of a warp are skipped by
// that warp; V rows past the sequence end are cleared in registers before P V.
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
constexpr int kMqTile = 64;        // KV tokens per stage and rows per CTA
constexpr int kMqStages = 3;
constexpr long long kMqWaitCycles = 4000000000LL;
#define kNegInfQ (-__int_as_float(0x7f800000))

// Address of 16-byte chunk `dch` of token row `row` when each 64-column half
// of the head dim is its own [64 rows][128 B] region with the 128-byte
// swizzle: 8 consecutive rows at one chunk hit 8 different bank groups.
__device__ __forceinline__ uint32_t swz_split(uint32_t base, int row, int dch) {
  return base + (dch >> 3) * (kMqTile * 128) + row * 128 + (((dch & 7) ^ (row & 7)) << 4);
}

// Producer warp: fill the ring with the KV tiles [0, ntiles) of (sequence,
// kv head): lane p issues the TMA loads of the tile's block-piece p.
// SPLIT: the stage holds each 64-column half of the head dim as its own
// [64 rows][128 B] region (one 3-D box per half); otherwise whole rows (one
// 4-D box).
template <int ROW_BYTES, int KV_BYTES, int STAGE_BYTES, bool SPLIT>
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
      if (SPLIT) {
        const uint32_t base = smem0 + st * STAGE_BYTES + lane * R * 128;
#pragma unroll
        for (int h = 0; h < ROW_BYTES / 128; ++h) {
          tma_load_3d(base + h * kMqTile * 128, tmK, h * 64, y, z, bar0 + 8u * st);
          tma_load_3d(base + KV_BYTES + h * kMqTile * 128, tmV, h * 64, y, z, bar0 + 8u * st);
        }
      } else {
        tma_load_4d(kdst, tmK, 0, 0, y, z, bar0 + 8u * st);
        tma_load_4d(kdst + KV_BYTES, tmV, 0, 0, y, z, bar0 + 8u * st);
      }
    }
    issued = i + 1;
  }
  if (lane == 0)
    for (int j = issued > kMqStages ? issued - kMqStages : 0; j < issued; ++j)
      mbar_wait_bounded(bar0 + 8u * (j % kMqStages), (j / kMqStages) & 1, abort_flag,
                        kMqWaitCycles);
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kMqThreads, 2)
multi_query_kernel(const MultiQueryArgs a, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV) {
  constexpr int HALVES = D / 64;
  constexpr int ROW_BYTES = HALVES * 128;
  constexpr int KV_BYTES = kMqTile * ROW_BYTES;
  constexpr int STAGE_BYTES = 2 * KV_BYTES;
  constexpr int KSTEPS = D / 16;        // k-steps of Q K^T
  constexpr int DN = D / 8;             // 8-wide head-dim tiles of O

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kMqStages * STAGE_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kMqStages);
  unsigned* tile_mask = reinterpret_cast<unsigned*>(bars + 2 * kMqStages) + 1;
  const uint32_t smem0 = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);

  const int s = blockIdx.z, kvh = blockIdx.y;
  const int row_tiles = (a.max_query_len * G + kMqTile - 1) / kMqTile;
  const int qt = blockIdx.x % row_tiles, split = blockIdx.x / row_tiles;
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
  const int r0 = qt * kMqTile;                       // first row of this CTA
  if (r0 >= n * G) return;
  const int i_last = min(n - 1, (r0 + kMqTile - 1) / G);
  const int kv_all = L - n + i_last + 1;             // keys any row here may see
  const int kv_lo = split * a.partition;             // this CTA's partition
  if (kv_lo >= kv_all) return;
  const int kv_end = min(kv_all, kv_lo + a.partition);
  const int ntiles = (kv_end - kv_lo + kMqTile - 1) / kMqTile;
  const int32_t* trow = a.tables + (int64_t)s * a.table_stride;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kMqStages; ++st) {
      mbar_init(bar0 + 8u * st, 1);
      mbar_init(bar0 + 8u * (kMqStages + st), kMqConsumers);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == kMqConsumers) {
    mq_produce<ROW_BYTES, KV_BYTES, STAGE_BYTES, true>(a, &tmK, &tmV, trow, kvh, kv_lo, kv_end,
                                                       ntiles,
                                                 smem0, bar0, tile_mask, abort_flag, lane);
    __syncthreads();
    if (*abort_flag && lane == 0) latch(a.err, PA_ERR_TIMEOUT);
    return;
  }

  // ---- consumer warp: rows rw0 .. rw0+15; this lane holds rows n8 and n8+8
  const int c = lane & 3, n8 = lane >> 2;
  const int rw0 = r0 + warp * 16;
  int pos[2];            // causal limit (last visible key) per held row; -1 = no row
  bool rv[2];
  uint32_t qa[KSTEPS][4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = rw0 + n8 + 8 * h;
    const int i = r / G;
    rv[h] = i < n;
    pos[h] = rv[h] ? L - n + i : -1;
  }
  {
    const T* qb[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = rw0 + n8 + 8 * h;
      qb[h] = reinterpret_cast<const T*>(a.q) +
              ((int64_t)(q0 + r / G) * Hq + (int64_t)kvh * G + r % G) * D;
    }
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        qa[ks][h] = rv[h] ? *reinterpret_cast<const uint32_t*>(qb[h] + ks * 16 + 2 * c) : 0u;
        qa[ks][h + 2] =
            rv[h] ? *reinterpret_cast<const uint32_t*>(qb[h] + ks * 16 + 8 + 2 * c) : 0u;
      }
    }
  }
  // the largest causal limit among this warp's 16 rows
  int warp_last = max(pos[0], pos[1]);
#pragma unroll
  for (int off = 1; off < 32; off <<= 1)
    warp_last = max(warp_last, __shfl_xor_sync(0xffffffffu, warp_last, off));

  float o[DN][4];
#pragma unroll
  for (int j = 0; j < DN; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m[2] = {kNegInfQ, kNegInfQ}, l[2] = {0.f, 0.f};
  const float sl2 = a.scale * kLog2e;
  const int B = a.block_size;
  const int R = B < kMqTile ? B : kMqTile;
  const int npieces = kMqTile / R;
  const unsigned full_mask = npieces >= 32 ? 0xffffffffu : ((1u << npieces) - 1u);

  for (int i = 0; i < ntiles; ++i) {
    const int st = i % kMqStages;
    if (!mbar_wait_bounded(bar0 + 8u * st, (i / kMqStages) & 1, abort_flag, kMqWaitCycles))
      break;
    const int ts = kv_lo + i * kMqTile;
    const int te = min(kv_end, ts + kMqTile);
    const uint32_t kst = smem0 + st * STAGE_BYTES;
    const uint32_t vst = kst + KV_BYTES;
    const unsigned pm = tile_mask[st];
    const bool need_zero = !(te - ts == kMqTile && pm == full_mask);
    if (ts <= warp_last) {
      float sacc[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
      for (int kp = 0; kp < KSTEPS / 2; ++kp) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          uint32_t kb[4];
          ldsm_x4(kb, swz_split(kst, nt * 8 + (lane & 7), 4 * kp + (lane >> 3)));
          MmaOps<T>::mma(sacc[nt], qa[2 * kp], kb[0], kb[1]);
          MmaOps<T>::mma(sacc[nt], qa[2 * kp + 1], kb[2], kb[3]);
        }
      }
      float mx[2] = {kNegInfQ, kNegInfQ};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int rr = nt * 8 + 2 * c + (e & 1);
          const int j = ts + rr;
          const int h = e >> 1;
          const bool ok = j <= pos[h] && j < te && ((pm >> (rr / R)) & 1u);
          sacc[nt][e] = ok ? sacc[nt][e] * sl2 : kNegInfQ;
          mx[h] = fmaxf(mx[h], sacc[nt][e]);
        }
      }
      float al[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        const float mn = fmaxf(m[h], mx[h]);
        const bool live = mn != kNegInfQ;
        al[h] = live ? exp2f(m[h] - mn) : 1.f;
        m[h] = mn;
        l[h] *= al[h];
      }
      uint32_t pa[4][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = e >> 1;
          p[e] = (m[h] != kNegInfQ) ? exp2f(sacc[nt][e] - m[h]) : 0.f;
        }
        const uint32_t lo = MmaOps<T>::pack(p[0], p[1]);   // row n8
        const uint32_t hi = MmaOps<T>::pack(p[2], p[3]);   // row n8 + 8
        const float2 flo = MmaOps<T>::unpack(lo), fhi = MmaOps<T>::unpack(hi);
        l[0] += flo.x + flo.y;
        l[1] += fhi.x + fhi.y;
        pa[nt >> 1][(nt & 1) * 2 + 0] = lo;
        pa[nt >> 1][(nt & 1) * 2 + 1] = hi;
      }
#pragma unroll
      for (int j = 0; j < DN; ++j) {
        o[j][0] *= al[0]; o[j][1] *= al[0]; o[j][2] *= al[1]; o[j][3] *= al[1];
      }
      // V rows that hold no token of this sequence may contain anything (NaN
      // included); their weight is 0, but 0 * NaN is NaN, so the fragment
      // halves of those rows are cleared in registers before the product.
      uint32_t vm[4][2];
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int rr = kt * 16 + hh * 8 + 2 * c;
          const bool v0 = !need_zero || ((ts + rr < te) && ((pm >> (rr / R)) & 1u));
          const bool v1 = !need_zero || ((ts + rr + 1 < te) && ((pm >> ((rr + 1) / R)) & 1u));
          vm[kt][hh] = (v0 ? 0x0000ffffu : 0u) | (v1 ? 0xffff0000u : 0u);
        }
      }
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
#pragma unroll
        for (int dp = 0; dp < DN / 2; ++dp) {
          uint32_t vb[4];
          ldsm_x4_trans(vb, swz_split(vst, kt * 16 + ((lane >> 3) & 1) * 8 + (lane & 7),
                                      2 * dp + (lane >> 4)));
          vb[0] &= vm[kt][0]; vb[1] &= vm[kt][1]; vb[2] &= vm[kt][0]; vb[3] &= vm[kt][1];
          MmaOps<T>::mma(o[2 * dp], pa[kt], vb[0], vb[1]);
          MmaOps<T>::mma(o[2 * dp + 1], pa[kt], vb[2], vb[3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar0 + 8u * (kMqStages + st));
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
  }
  __syncthreads();
  if (*abort_flag) return;
  T* out = reinterpret_cast<T*>(a.out);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (!rv[h]) continue;
    const int r = rw0 + n8 + 8 * h;
    const int64_t t = q0 + r / G;
    const int head = kvh * G + r % G;
    const int count = (pos[h] + a.partition) / a.partition;   // partitions holding its keys
    if (count == 1) {
      if (split != 0) continue;
      const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
      T* op = out + (t * Hq + head) * D;
#pragma unroll
      for (int j = 0; j < DN; ++j) {
        const uint32_t v = MmaOps<T>::pack(o[j][2 * h] * inv, o[j][2 * h + 1] * inv);
        *reinterpret_cast<uint32_t*>(op + j * 8 + 2 * c) = v;
      }
    } else if (split < count) {
      const int64_t slot = (t * Hq + head) * a.num_splits + split;
      float* acc = a.ws_acc + slot * D;
#pragma unroll
      for (int j = 0; j < DN; ++j)
        *reinterpret_cast<float2*>(acc + j * 8 + 2 * c) = make_float2(o[j][2 * h], o[j][2 * h + 1]);
      if (c == 0) {
        a.ws_ml[2 * slot] = m[h];
        a.ws_ml[2 * slot + 1] = l[h];
      }
    }
  }
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
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
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
    mq_produce<ROW_BYTES, KV_BYTES, STAGE_BYTES, false>(a, &tmK, &tmV, trow, kvh, kv_lo, kv_end,
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
          float p[4], al[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float mn = fmaxf(m[nt][e], mx[e]);
            const bool live = mn != kNegInfQ;
            al[e] = live ? exp2f(m[nt][e] - mn) : 1.f;
            p[e] = live ? exp2f(x[e] - mn) : 0.f;
            p[e + 2] = live ? exp2f(x[e + 2] - mn) : 0.f;
            m[nt][e] = mn;
          }
          const uint32_t cA = MmaOps<T>::pack(p[0], p[1]);
          const uint32_t cB = MmaOps<T>::pack(p[2], p[3]);
          const float2 fA = MmaOps<T>::unpack(cA), fB = MmaOps<T>::unpack(cB);
          l[nt][0] = l[nt][0] * al[0] + fA.x + fB.x;
          l[nt][1] = l[nt][1] * al[1] + fA.y + fB.y;
#pragma unroll
          for (int mt = 0; mt < KSTEPS; ++mt) {
            o[nt][mt][0] *= al[0]; o[nt][mt][1] *= al[1];
            o[nt][mt][2] *= al[0]; o[nt][mt][3] *= al[1];
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

PFN_cuTensorMapEncodeTiled_v12000 g_encode_halves = nullptr;
std::once_flag g_encode_halves_once;

// Pool [NB][Hkv][B][D] (16-bit dtype) as a 3-D tensor {D, B, NB*Hkv} with
// boxes of one 64-column half of min(B, 64) rows, 128-byte swizzle.
bool encode_pool_halves_map(CUtensorMap* map, const void* base, int dtype, int64_t num_blocks,
                            int num_kv_heads, int block_size, int head_size) {
  std::call_once(g_encode_halves_once, []() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode_halves = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode_halves) return false;
  const uint64_t D = head_size, B = block_size;
  const uint64_t planes = (uint64_t)num_blocks * num_kv_heads;
  if (planes == 0 || planes > 0x7fffffffull || D % 64 != 0) return false;
  cuuint64_t dims[3] = {D, B, planes};
  cuuint64_t strides[2] = {D * 2, B * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)(B < 64 ? B : 64), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode_halves(map,
                         dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         3, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
constexpr int mq_smem_bytes() {
  return 1024 + kMqStages * 2 * kMqTile * (D / 64) * 128 + 2 * kMqStages * 8 + 4 +
         4 * kMqStages + 16;
}

template <typename T, int D, int G>
cudaError_t launch_mq_tdg(const MultiQueryArgs& a, cudaStream_t st) {
  const int64_t rows_ = (int64_t)a.max_query_len * G;
  const bool cols_kernel = (rows_ + kMqsCols - 1) / kMqsCols <= 2;
  // the row kernel reads every K/V row many times: conflict-free halves; the
  // column kernel streams: whole-row boxes
  CUtensorMap tk, tv;
  const bool ok =
      cols_kernel
          ? encode_kv_pool_map(&tk, a.kc, a.dtype, a.num_blocks, a.num_kv_heads, a.block_size,
                               a.head_size) &&
                encode_kv_pool_map(&tv, a.vc, a.dtype, a.num_blocks, a.num_kv_heads,
                                   a.block_size, a.head_size)
          : encode_pool_halves_map(&tk, a.kc, a.dtype, a.num_blocks, a.num_kv_heads,
                                   a.block_size, a.head_size) &&
                encode_pool_halves_map(&tv, a.vc, a.dtype, a.num_blocks, a.num_kv_heads,
                                       a.block_size, a.head_size);
  if (!ok) return cudaErrorInvalidValue;
  constexpr int smem = mq_smem_bytes<D>();
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, []() {
    attr = cudaFuncSetAttribute(multi_query_kernel<T, D, G>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (attr != cudaSuccess) return attr;
  const int64_t rows = (int64_t)a.max_query_len * G;
  const int64_t tiles = (rows + kMqTile - 1) / kMqTile;
  if (tiles == 0 || a.num_seqs == 0) return cudaSuccess;
  const int64_t col_tiles = (rows + kMqsCols - 1) / kMqsCols;
  if (col_tiles <= 2) {
    // a few new tokens per sequence: columns as N, KV tokens as M
    static std::once_flag once_cols;
    static cudaError_t attr_cols = cudaSuccess;
    std::call_once(once_cols, []() {
      attr_cols = cudaFuncSetAttribute(multi_query_cols_kernel<T, D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr_cols != cudaSuccess) return attr_cols;
    dim3 grid((unsigned)(col_tiles * a.num_splits), a.num_kv_heads, a.num_seqs);
    multi_query_cols_kernel<T, D, G><<<grid, kMqThreads, smem, st>>>(a, tk, tv);
  } else if (rows > kMqTile) {
    // long runs (prefill chunks): the tcgen05 kernel, 128 rows per CTA
    cudaError_t e = launch_multi_query_tc(a, st);
    if (e != cudaSuccess) return e;
  } else {
    dim3 grid((unsigned)(tiles * a.num_splits), a.num_kv_heads, a.num_seqs);
    multi_query_kernel<T, D, G><<<grid, kMqThreads, smem, st>>>(a, tk, tv);
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
