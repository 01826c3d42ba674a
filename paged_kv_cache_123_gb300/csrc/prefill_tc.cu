// Causal paged attention for runs of more than 16 (token, head) rows per KV
// head (prefill chunks, speculative runs) on the fifth-generation tensor
// cores: tcgen05.mma with fp32 accumulators, scores and softmax weights in
// tensor memory (TMEM).
//
// What is computed is the multi-query attention of prefill_mma.cu: new token
// i of sequence s (n_s new tokens, L_s tokens in the pool including them)
// sits at position L_s - n_s + i and attends to positions 0 .. L_s - n_s + i
// through the block table ("vLLM 的 PagedAttention：显存管理如何撑起大模型推理"
// §2.5: one token budget covers prefill chunks; "PagedAttention 核心创新深度
// 分析" §2.3: the slot mapping places any number of tokens per request).
//
// One CTA owns 128 rows — (new token, query head) pairs of one KV head,
// query-major — and walks its causal KV range in tiles of 128 tokens:
//   * producer warps load the CTA's Q tile once (3-D TMA straight from the
//     [tokens][heads][D] query tensor) and the K and V tiles by 3-D TMA
//     boxes of one 64-column half of one block's rows (128-byte swizzle),
//     into a three-stage K ring and a two-stage V ring; a K stage is
//     released as soon as S of its tile is computed, a V stage when P V is;
//   * one thread of the MMA warp issues S = Q K^T (M = 128 rows, N = 128
//     tokens, K = D; both operands in shared memory) into one of two TMEM
//     score buffers and [O | l] += P [V | 1] (M = 128, N = D + 16, K = 128
//     tokens) with P read from TMEM and V read N-major straight from its
//     token rows; each V stage carries a constant group of ones after the
//     head dims, so column D of the output holds the row sums of exactly
//     the rounded weights; each group of MMAs completes on an mbarrier
//     (tcgen05.commit). P of tile j lives in score buffer j&1, so S of tile
//     j+2 follows the completion of P V of tile j, while the softmax warps
//     work on tile j+1;
//   * eight softmax warps, two warpgroups, own half a row each per thread
//     (TMEM lane = row; warpgroup h takes score columns 64h .. 64h+63): they
//     read the scores with tcgen05.ld, apply the causal limit and the scale
//     in the log2 domain, exchange the two half-row maxima through shared
//     memory, and write P (16-bit) over their own scores with tcgen05.st.
//     Output and sums in TMEM are rescaled only when a row's running
//     maximum grew by more than 2^8 (the weights stay below 256, and the
//     final division uses the same reference); only then does a softmax
//     warp wait for the previous tile's P V.
// Keeping S and P out of shared memory leaves its bandwidth to the K/V
// operands and their TMA loads.
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "launchers.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace pa {
namespace {

constexpr int kTcRows = 128;              // query rows per CTA (MMA M)
constexpr int kTcKv = 128;                // KV tokens per tile
constexpr int kTcStages = 3;              // K ring depth
constexpr int kTcVStages = 2;             // V ring depth
constexpr int kTcSoftmaxWarps = 8;        // two warpgroups: columns 0-63, 64-127
constexpr int kTcKProducerWarp = 8;       // Q and K tiles
constexpr int kTcMmaWarp = 9;
constexpr int kTcVProducerWarp = 10;      // V tiles
constexpr int kTcThreads = 11 * 32;
constexpr int kTcCols = kTcKv / 2;        // score columns per softmax thread
// TMEM columns: score buffers S0 [0,128) and S1 [128,256), O [256, 256+D)
// and the row sums l in column 256+D (the ones group of V, 16 columns). The
// 16-bit weights P of tile j overwrite the scores of their own half row in
// buffer j&1 (half h: columns 64h .. 64h+31 of the buffer)
constexpr uint32_t kTcTmemCols = 512;
constexpr uint32_t kTcOCol = 256;
constexpr long long kTcWaitCycles = 4000000000LL;
constexpr float kTcRescaleLog2 = 8.f;
#define kNegInfT (-__int_as_float(0x7f800000))

template <int D>
struct TcLayout {
  static constexpr int HALVES = D / 64;
  static constexpr int HALF_BYTES = kTcRows * 128;          // 128 rows x 64 columns
  static constexpr int Q_BYTES = HALVES * HALF_BYTES;
  static constexpr int KV_HALF = kTcKv * 128;
  static constexpr int KV_BYTES = HALVES * KV_HALF;         // one K (or V) tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + Q_BYTES;
  static constexpr int V_OFF = K_OFF + kTcStages * KV_BYTES;
  // a V stage is the tile's 64-column groups of the head dim plus one group
  // of 16-bit ones: P x [V | 1] also gives the row sums of the weights
  static constexpr int V_STAGE = KV_BYTES + KV_HALF;
  static constexpr int BAR_OFF = V_OFF + kTcVStages * V_STAGE;
  // q_full, k_full[3], k_empty[3], v_full[3], v_empty[3], s_full[2], p_full,
  // o_done, done
  static constexpr int NBARS = 18;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;     // tmem base, abort flag
  // row maxima and row sums exchanged between the two softmax warpgroups
  static constexpr int XCH_OFF = MISC_OFF + 32;            // float [2][128]
  static constexpr int SMEM = XCH_OFF + 2 * kTcRows * 4 + 1024;   // + alignment slack
  static_assert(SMEM <= 232448, "over the shared memory of one CTA");
};

enum : int {
  kBarQ = 0, kBarKFull = 1, kBarKEmpty = 4, kBarVFull = 7, kBarVEmpty = 10,
  kBarSFull = 13, kBarPFull = 15, kBarODone = 16, kBarDone = 17
};

// max of three floats (one instruction)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (a0, a1) * s + t for a pair, one packed f32x2 instruction
__device__ __forceinline__ void fma2(float a0, float a1, float s, float t, float& d0, float& d1) {
  uint64_t a, m, c, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(m) : "f"(s));
  asm("mov.b64 %0, {%1, %1};" : "=l"(c) : "f"(t));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(m), "l"(c));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
}

// Barrier 1 over the eight softmax warps (256 threads) that also returns
// whether every one of them passed `ok`, so they leave their loop together.
__device__ __forceinline__ bool softmax_bar_and(bool ok) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n"
      " barrier.cta.red.and.pred po, 1, 256, pi;\n selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(out) : "r"((uint32_t)ok) : "memory");
  return out != 0;
}

// 2^x by the SFU's ex2.approx (inputs here are <= 8; -inf gives +0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// two fp32 values packed to the 16-bit input type (round to nearest)
template <typename T>
struct Pack2;
template <>
struct Pack2<__nv_bfloat16> {
  __device__ __forceinline__ static uint32_t pack_out(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};
template <>
struct Pack2<__half> {
  __device__ __forceinline__ static uint32_t pack_out(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

// Block pieces of tile [ts, te): piece p = R = min(B, 128) rows of one
// block; bit p set when its table entry names a block of the pool.
__device__ __forceinline__ unsigned tc_piece_mask(const MultiQueryArgs& a, const int32_t* trow,
                                                  int ts, int te, int lane, int64_t* blk_out) {
  const int B = a.block_size;
  const int R = B < kTcKv ? B : kTcKv;
  const int tok = ts + lane * R;
  int64_t blk = -1;
  bool mine = false;
  if (lane < kTcKv / R && tok < te) {
    blk = trow[tok >> (__ffs(B) - 1)];
    mine = blk >= 0 && blk < a.num_blocks;
  }
  *blk_out = blk;
  return __ballot_sync(0xffffffffu, mine);
}

// Producer warp for one operand (K, with the Q tile first, or V): the tiles
// of [kv_lo, kv_end) into that operand's ring. Lane p loads piece p of a
// tile, both 64-column halves.
template <int D, bool IS_V>
__device__ void tc_produce(const MultiQueryArgs& a, const CUtensorMap* tmQ,
                           const CUtensorMap* tm, const int32_t* trow, int kvh, int q_tok,
                           int kv_lo, int kv_end, int ntiles, uint32_t s0, uint32_t bar,
                           volatile int* abort_flag, int lane, int G) {
  using Ly = TcLayout<D>;
  const int full = IS_V ? kBarVFull : kBarKFull;
  const int empty = IS_V ? kBarVEmpty : kBarKEmpty;
  constexpr int NST = IS_V ? kTcVStages : kTcStages;
  constexpr int STRIDE = IS_V ? Ly::V_STAGE : Ly::KV_BYTES;
  const uint32_t base = s0 + (IS_V ? Ly::V_OFF : Ly::K_OFF);
  if (lane == 0) {
    prefetch_tensormap(tm);
    if (!IS_V) {
      prefetch_tensormap(tmQ);
      mbar_arrive_expect_tx(bar + 8u * kBarQ, (uint32_t)Ly::Q_BYTES);
#pragma unroll
      for (int h = 0; h < Ly::HALVES; ++h)
        tma_load_3d(s0 + Ly::Q_OFF + h * Ly::HALF_BYTES, tmQ, h * 64, kvh * G, q_tok,
                    bar + 8u * kBarQ);
    }
  }
  const int B = a.block_size;
  const int R = B < kTcKv ? B : kTcKv;
  int issued = 0;
  for (int i = 0; i < ntiles; ++i) {
    const int st = i % NST;
    const int ts = kv_lo + i * kTcKv;
    const int te = min(kv_end, ts + kTcKv);
    int64_t blk;
    const unsigned pm = tc_piece_mask(a, trow, ts, te, lane, &blk);
    const bool mine = (pm >> lane) & 1u;
    if (!IS_V && lane < kTcKv / R && ts + lane * R < te && !mine)
      latch(a.err, PA_ERR_OUT_OF_RANGE);
    int ok = 1;
    if (lane == 0) {
      if (i >= NST)
        ok = mbar_wait_bounded(bar + 8u * (empty + st), ((i / NST) - 1) & 1, abort_flag,
                               kTcWaitCycles);
      if (ok)
        mbar_arrive_expect_tx(bar + 8u * (full + st),
                              (uint32_t)__popc(pm) * (uint32_t)R * (uint32_t)(D * 2));
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) break;
    if (mine) {
      const int z = (int)(blk * a.num_kv_heads + kvh);
      const int y = (ts + lane * R) & (B - 1);
      const uint32_t d = base + st * STRIDE + lane * R * 128;
#pragma unroll
      for (int h = 0; h < Ly::HALVES; ++h)
        tma_load_3d(d + h * Ly::KV_HALF, tm, h * 64, y, z, bar + 8u * (full + st));
    }
    issued = i + 1;
  }
  // let this warp's copies land before the CTA can leave (also after a
  // timeout: these waits have their own limit and ignore the abort flag)
  if (lane == 0) {
    if (!IS_V) mbar_wait_drain(bar + 8u * kBarQ, 0, kTcWaitCycles);
    for (int j = issued > NST ? issued - NST : 0; j < issued; ++j)
      mbar_wait_drain(bar + 8u * (full + j % NST), (j / NST) & 1, kTcWaitCycles);
  }
}

// MMA issue (one thread): S_j = Q K_j^T into TMEM score buffer j&1, and
// [O | l] += P_j [V_j | 1] (P_j from the same buffer) once the softmax warps
// have written P_j. S_{j+2} reuses the buffer, so it is issued once P_j V_j
// has completed; S_{j+1} is already in place for the softmax warps.
template <typename T, int D>
__device__ void tc_issue(int ntiles, uint32_t s0, uint32_t bar, uint32_t tmem,
                         volatile int* abort_flag) {
  using Ly = TcLayout<D>;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t idS = idesc_f16(kBf16, kTcRows, kTcKv, false, false);
  constexpr uint32_t idO = idesc_f16(kBf16, kTcRows, D + 16, false, true);
  const uint32_t qa = s0 + Ly::Q_OFF;
  auto issue_pv = [&](int t) -> bool {
    const int vs = t % kTcVStages;
    if (!mbar_wait_bounded(bar + 8u * kBarPFull, t & 1, abort_flag, kTcWaitCycles)) return false;
    if (!mbar_wait_bounded(bar + 8u * (kBarVFull + vs), (t / kTcVStages) & 1, abort_flag,
                           kTcWaitCycles))
      return false;
    tc_fence_after();
    const uint32_t vb = s0 + Ly::V_OFF + vs * Ly::V_STAGE;
    const uint32_t pt = tmem + (uint32_t)(t & 1) * kTcKv;
#pragma unroll
    for (int ks = 0; ks < kTcKv / 16; ++ks) {
      // [V | 1] tile: token rows of 64 columns per 128-byte line (N-major);
      // 16 tokens per k-step, the next 64-column group at KV_HALF. P of
      // tokens 16 ks .. 16 ks + 15: half ks / 4 of the row, 8 columns
      const uint64_t bd = smem_desc_sw128(vb + ks * 2048, Ly::KV_HALF, 1024);
      mma_f16_ts(tmem + kTcOCol, pt + (ks >> 2) * kTcCols + (ks & 3) * 8, bd, idO,
                 (t > 0 || ks > 0) ? 1u : 0u);
    }
    mma_commit(bar + 8u * kBarODone);
    mma_commit(bar + 8u * (kBarVEmpty + vs));
    return true;
  };
  // S_t into score buffer t&1 once K_t has landed (the caller has seen
  // P_{t-2} V_{t-2} complete, so nothing reads the buffer any more)
  auto issue_s = [&](int t) -> bool {
    const int sb = t & 1, ks_ = t % kTcStages;
    if (!mbar_wait_bounded(bar + 8u * (kBarKFull + ks_), (t / kTcStages) & 1, abort_flag,
                           kTcWaitCycles))
      return false;
    tc_fence_after();
    const uint32_t kb = s0 + Ly::K_OFF + ks_ * Ly::KV_BYTES;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint64_t ad = smem_desc_sw128(qa + (ks >> 2) * Ly::HALF_BYTES + (ks & 3) * 32, 16, 1024);
      const uint64_t bd = smem_desc_sw128(kb + (ks >> 2) * Ly::KV_HALF + (ks & 3) * 32, 16, 1024);
      mma_f16_ss(tmem + sb * kTcKv, ad, bd, idS, ks > 0 ? 1u : 0u);
    }
    mma_commit(bar + 8u * (kBarSFull + sb));
    mma_commit(bar + 8u * (kBarKEmpty + ks_));
    return true;
  };
  // the softmax warps work on tile j+1 while P_j V_j and then S_{j+2} run
  bool ok = mbar_wait_bounded(bar + 8u * kBarQ, 0, abort_flag, kTcWaitCycles);
  for (int t = 0; ok && t < 2 && t < ntiles; ++t) ok = issue_s(t);
  for (int j = 0; ok && j < ntiles; ++j) {
    ok = issue_pv(j);
    if (ok && j + 2 < ntiles) {
      ok = mbar_wait_bounded(bar + 8u * kBarODone, j & 1, abort_flag, kTcWaitCycles);
      if (ok) ok = issue_s(j + 2);
    }
  }
  // every MMA issued above has completed once this barrier fires (waited
  // for also after a timeout, before the CTA frees its TMEM)
  mma_commit(bar + 8u * kBarDone);
  mbar_wait_drain(bar + 8u * kBarDone, 0, kTcWaitCycles);
}

// SKIP_IDLE: runs shorter than a row tile leave whole warps without a token
// row; that instantiation lets such warps skip the score work.
template <typename T, int D, int G, bool SKIP_IDLE>
__global__ void __launch_bounds__(kTcThreads, 1)
multi_query_tc_kernel(const MultiQueryArgs a, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV) {
  using Ly = TcLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, reached by pointer arithmetic on the shared
  // array itself so the compiler keeps every access in the shared space
  // (an integer round trip would make them generic loads)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t s0 = smem_u32(smem);
  const uint32_t bar = s0 + Ly::BAR_OFF;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Ly::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

  const int s = blockIdx.z, kvh = blockIdx.y;
  const int row_tiles = (a.max_query_len * G + kTcRows - 1) / kTcRows;
  const int qt = row_tiles - 1 - (int)(blockIdx.x % row_tiles);   // longest rows first
  const int split = (int)(blockIdx.x / row_tiles);
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
  const int r0 = qt * kTcRows;                      // first row of this CTA
  if (r0 >= n * G) return;
  const int i_last = min(n - 1, (r0 + kTcRows - 1) / G);
  const int kv_all = L - n + i_last + 1;            // keys any row here may see
  const int kv_lo = split * a.partition;
  if (kv_lo >= kv_all) return;
  const int kv_end = min(kv_all, kv_lo + a.partition);
  const int ntiles = (kv_end - kv_lo + kTcKv - 1) / kTcKv;

  if (threadIdx.x == 0) {
    mbar_init(bar + 8u * kBarQ, 1);
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(bar + 8u * (kBarKFull + i), 1);
      mbar_init(bar + 8u * (kBarKEmpty + i), 1);
      mbar_init(bar + 8u * (kBarVFull + i), 1);
      mbar_init(bar + 8u * (kBarVEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(bar + 8u * (kBarSFull + i), 1);
    mbar_init(bar + 8u * kBarPFull, kTcSoftmaxWarps);
    mbar_init(bar + 8u * kBarODone, 1);
    mbar_init(bar + 8u * kBarDone, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kTcMmaWarp) {
    tmem_alloc(s0 + Ly::MISC_OFF, kTcTmemCols);
    tmem_relinquish();
  }
  {
    // the ones group of every V stage (1.0 in either 16-bit type); TMA never
    // writes it
    const uint32_t one2 = std::is_same<T, __nv_bfloat16>::value ? 0x3f803f80u : 0x3c003c00u;
    for (int i = threadIdx.x; i < kTcVStages * Ly::KV_HALF / 16; i += kTcThreads) {
      const int st = i / (Ly::KV_HALF / 16), off = i % (Ly::KV_HALF / 16);
      asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};"
                   ::"r"(s0 + Ly::V_OFF + st * Ly::V_STAGE + Ly::KV_BYTES + off * 16), "r"(one2)
                   : "memory");
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  const int32_t* trow = a.tables + (int64_t)s * a.table_stride;
  if (warp == kTcKProducerWarp) {
    tc_produce<D, false>(a, &tmQ, &tmK, trow, kvh, q0 + r0 / G, kv_lo, kv_end, ntiles, s0, bar,
                         abort_flag, lane, G);
  } else if (warp == kTcVProducerWarp) {
    tc_produce<D, true>(a, &tmQ, &tmV, trow, kvh, q0 + r0 / G, kv_lo, kv_end, ntiles, s0, bar,
                        abort_flag, lane, G);
  } else if (warp == kTcMmaWarp) {
    if (lane == 0) tc_issue<T, D>(ntiles, s0, bar, tmem, abort_flag);
    __syncwarp();
  } else {
    // ---- softmax warps: thread = (half hf, row r); TMEM lane r, score
    // columns 64 hf .. 64 hf + 63
    const int hf = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const int rr = r0 + r;
    const int i = rr / G;
    const bool rv = i < n;
    const int pos = rv ? L - n + i : -1;            // causal limit of this row
    // a warp none of whose rows holds a token (short runs: 4 tokens x 8
    // heads fill 32 of the 128 rows) skips the score work; its P rows are
    // written as zeros once and its V-row clearing duty stays
    const bool idle = SKIP_IDLE && __all_sync(0xffffffffu, !rv);
    const float sl2 = a.scale * kLog2e;
    const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
    float* xch = reinterpret_cast<float*>(smem + Ly::XCH_OFF);   // [2 halves][128]
    const int B = a.block_size;
    const int R = B < kTcKv ? B : kTcKv;
    const int rshift = __ffs(R) - 1;
    const int npieces = kTcKv / R;
    const unsigned full_mask = npieces >= 32 ? 0xffffffffu : ((1u << npieces) - 1u);
    // table entry of this lane's block piece of tile t (-1: none), read one
    // tile ahead so its latency hides behind the current tile
    auto piece_entry = [&](int t) -> int {
      const int ts = kv_lo + t * kTcKv;
      const int tok = ts + lane * R;
      if (lane < npieces && tok < min(kv_end, ts + kTcKv))
        return trow[tok >> (__ffs(B) - 1)];
      return -1;
    };
    int ent_next = piece_entry(0);
    float m_use = kNegInfT;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int sb = j & 1;
      const int ts = kv_lo + j * kTcKv;
      const int te = min(kv_end, ts + kTcKv);
      const int ent = ent_next;
      if (j + 1 < ntiles) ent_next = piece_entry(j + 1);
      // block pieces of the tile that exist (the producers load exactly these)
      const unsigned pm = __ballot_sync(0xffffffffu, ent >= 0 && ent < a.num_blocks);
      if (ok)
        ok = mbar_wait_bounded(bar + 8u * (kBarSFull + sb), (j >> 1) & 1, abort_flag,
                               kTcWaitCycles);
      // tcgen05.ld / st are warp-collective: the whole warp goes on or stops
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      const bool whole = (pm == full_mask) && (te - ts == kTcKv);
      const int lim = min(pos, te - 1) - ts - hf * kTcCols;   // last own column usable
      // valid own columns of 32-column chunk ch: causal / length limit and
      // loaded pieces
      auto chunk_mask = [&](int ch) -> uint32_t {
        const int c0 = ch * 32;
        uint32_t m = lim < c0 ? 0u : (lim >= c0 + 31 ? 0xffffffffu : ((2u << (lim - c0)) - 1u));
        if (!whole) {
          const int g0 = hf * kTcCols + c0;         // tile column of bit 0
          uint32_t pmask = 0;
          if (R >= 32) {
            pmask = ((pm >> (g0 >> rshift)) & 1u) ? 0xffffffffu : 0u;
          } else {
            for (int k = 0; k < 32 / R; ++k)
              if ((pm >> ((g0 >> rshift) + k)) & 1u) pmask |= ((1u << R) - 1u) << (k * R);
          }
          m &= pmask;
        }
        return m;
      };
      // interior tiles (every own column valid for every row of the warp)
      // skip the per-column masks. Rows that hold no token (a run shorter
      // than the row tile, e.g. 3 tokens x 8 heads = 24 of 32 rows) do not
      // count: an MMA row only feeds its own output row, which is never
      // written, so whatever their weights are (finite here: a whole tile
      // has no stale K rows) they change nothing
      const bool fast =
          __all_sync(0xffffffffu, whole && (lim >= kTcCols - 1 || !rv)) && sl2 > 0.f;
      const uint32_t sadr = tmem + lanes + sb * kTcKv + hf * kTcCols;
      // this thread's 64 scores, one load; they stay in registers for both
      // passes
      uint32_t v[kTcCols];
      if (ok && !idle) {
        tmem_ld64(sadr, v);
      } else if (SKIP_IDLE) {
#pragma unroll
        for (int e = 0; e < kTcCols; ++e) v[e] = 0u;
      }
      // positive scale (the usual case): the invalid scores of a boundary
      // tile become -inf in place, so both passes below run without masks
      // (-inf times the scale stays -inf, and 2^-inf is 0); a zero or
      // negative scale takes the general, per-element masked path
      const bool pscale = sl2 > 0.f;
      auto own_mask = [&](int ch) -> uint32_t { return fast ? 0xffffffffu : chunk_mask(ch); };
      if (ok && !idle && pscale && !fast && rv) {
#pragma unroll
        for (int ch = 0; ch < kTcCols / 32; ++ch) {
          const uint32_t m = chunk_mask(ch);
          if (m != 0xffffffffu) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (!((m >> e) & 1u)) v[ch * 32 + e] = __float_as_uint(kNegInfT);
          }
        }
      }
      // pass 1: maximum of the valid scaled scores of this half row
      float mx = kNegInfT;
      if (ok && !idle) {
        if (pscale) {
          float mx0 = kNegInfT, mx1 = kNegInfT;
#pragma unroll
          for (int e = 0; e < kTcCols; e += 4) {
            mx0 = fmax3(mx0, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
            mx1 = fmax3(mx1, __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
          }
          mx = fmaxf(mx0, mx1) * sl2;       // the scale is positive: max commutes
        } else {
#pragma unroll
          for (int ch = 0; ch < kTcCols / 32; ++ch) {
            const uint32_t m = own_mask(ch);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              mx = fmaxf(mx, ((m >> e) & 1u) ? __uint_as_float(v[ch * 32 + e]) * sl2 : kNegInfT);
          }
        }
      }
      // the two halves of the row meet: exchange the maxima; the second
      // barrier keeps the next tile's write behind this read
      xch[hf * kTcRows + r] = mx;
      ok = softmax_bar_and(ok);           // both warpgroups, all 256 threads
      if (!ok) break;
      mx = fmaxf(mx, xch[(hf ^ 1) * kTcRows + r]);
      asm volatile("bar.sync 1, 256;" ::: "memory");
      const float m_new = fmaxf(m_use, mx);
      float alpha = 1.f;
      bool resc = false;
      if (m_use == kNegInfT) {
        m_use = m_new;                  // nothing accumulated for this row yet
      } else if (m_new > m_use + kTcRescaleLog2) {
        alpha = exp2f(m_use - m_new);
        resc = true;
        m_use = m_new;
      }
      // pass 2: P = 2^(x - m_use) rounded to the input type, 16 columns of
      // packed pairs per 32 scores, over this thread's own (already loaded)
      // scores in buffer j&1 (both halves have passed the exchange barrier,
      // so every score of the buffer is in registers); the row sums come
      // from the MMA's ones group. Rows of idle warps get zeros every tile:
      // S of tile j+2 overwrites the buffer.
      const bool live = m_use != kNegInfT;
      const float nm = -m_use;
      const uint32_t padr = sadr;
      // tcgen05.st is warp-collective: the branch is taken by whole warps
      if (pscale && !idle && __all_sync(0xffffffffu, live)) {
#pragma unroll
        for (int ch = 0; ch < kTcCols / 32; ++ch) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float x0, x1;
            fma2(__uint_as_float(v[ch * 32 + e]), __uint_as_float(v[ch * 32 + e + 1]), sl2, nm,
                 x0, x1);
            pk[e >> 1] = Pack2<T>::pack_out(ex2_approx(x0), ex2_approx(x1));
          }
          tmem_st16(padr + ch * 16, pk);
        }
      } else {
#pragma unroll
        for (int ch = 0; ch < kTcCols / 32; ++ch) {
          uint32_t pk[16];
          if (idle) {
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = 0u;
          } else {
            const uint32_t vm = live ? own_mask(ch) : 0u;
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float x0, x1;
              fma2(__uint_as_float(v[ch * 32 + e]), __uint_as_float(v[ch * 32 + e + 1]), sl2,
                   nm, x0, x1);
              const float p0 = ((vm >> e) & 1u) ? ex2_approx(x0) : 0.f;
              const float p1 = ((vm >> (e + 1)) & 1u) ? ex2_approx(x1) : 0.f;
              pk[e >> 1] = Pack2<T>::pack_out(p0, p1);
            }
          }
          tmem_st16(padr + ch * 16, pk);
        }
      }
      // the output is rescaled only when some row of the warp needs it (the
      // other half row takes the same decision), after P V of tile j-1 has
      // completed (P V of tile j waits for this warp's P, so the phase is
      // current)
      if (__any_sync(0xffffffffu, resc)) {
        if (j >= 1) {
          ok = mbar_wait_bounded(bar + 8u * kBarODone, (j - 1) & 1, abort_flag, kTcWaitCycles);
          ok = __all_sync(0xffffffffu, ok);
          tc_fence_after();
        }
        if (ok) {
#pragma unroll 1
          for (int ch = 0; ch < D / 64; ++ch) {
            const uint32_t oadr = tmem + lanes + kTcOCol + hf * (D / 2) + ch * 32;
            uint32_t v[32];
            tmem_ld32(oadr, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st32(oadr, v);
          }
          if (hf == 0) {                // the row sums, once per row
            const uint32_t ladr = tmem + lanes + kTcOCol + D;
            tmem_st1(ladr, __float_as_uint(__uint_as_float(tmem_ld1(ladr)) * alpha));
          }
        }
      }
      // V rows that hold no token of this tile may contain anything (NaN
      // included) and 0 * NaN is NaN inside the MMA: clear them (row r, the
      // 64-column half hf of the head dim)
      if (!whole && ok && hf < Ly::HALVES) {
        // the V tile must have landed before its rows are cleared (its stage
        // is not refilled before P V of this tile, so the phase is current)
        const int vs = j % kTcVStages;
        ok = mbar_wait_bounded(bar + 8u * (kBarVFull + vs), (j / kTcVStages) & 1, abort_flag,
                               kTcWaitCycles);
        const bool row_ok = r < te - ts && ((pm >> (r >> rshift)) & 1u);
        if (ok && !row_ok) {
          const uint32_t vrow = s0 + Ly::V_OFF + vs * Ly::V_STAGE + hf * Ly::KV_HALF + r * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};"
                         ::"r"(vrow + k * 16), "r"(0u) : "memory");
        }
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar + 8u * kBarPFull);
    }
    if (ok && ntiles > 0) {
      // the MMA thread commits kBarDone after its last P V
      ok = mbar_wait_bounded(bar + 8u * kBarDone, 0, abort_flag, kTcWaitCycles);
      tc_fence_after();
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      const float l = __uint_as_float(tmem_ld1(tmem + lanes + kTcOCol + D));
      const int64_t t = q0 + i;
      const int head = kvh * G + rr % G;
      const int count = rv ? (pos + a.partition) / a.partition : 0;
      const bool direct = rv && count == 1 && split == 0;
      const bool partial = rv && count > 1 && split < count;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      T* out = reinterpret_cast<T*>(a.out);
      const int64_t slot = (t * Hq + head) * a.num_splits + split;
#pragma unroll 1
      for (int ch = 0; ch < D / 64; ++ch) {
        const int c0 = hf * (D / 2) + ch * 32;      // output columns c0 .. c0+31
        uint32_t v[32];
        tmem_ld32(tmem + lanes + kTcOCol + c0, v);
        if (direct) {
          uint4* op = reinterpret_cast<uint4*>(out + (t * Hq + head) * D + c0);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = Pack2<T>::pack_out(__uint_as_float(v[8 * q + 0]) * inv,
                                     __uint_as_float(v[8 * q + 1]) * inv);
            w.y = Pack2<T>::pack_out(__uint_as_float(v[8 * q + 2]) * inv,
                                     __uint_as_float(v[8 * q + 3]) * inv);
            w.z = Pack2<T>::pack_out(__uint_as_float(v[8 * q + 4]) * inv,
                                     __uint_as_float(v[8 * q + 5]) * inv);
            w.w = Pack2<T>::pack_out(__uint_as_float(v[8 * q + 6]) * inv,
                                     __uint_as_float(v[8 * q + 7]) * inv);
            op[q] = w;
          }
        } else if (partial) {
          float4* acc = reinterpret_cast<float4*>(a.ws_acc + slot * D + c0);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            acc[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        }
      }
      if (partial && hf == 0) {
        a.ws_ml[2 * slot] = m_use;
        a.ws_ml[2 * slot + 1] = l;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) latch(a.err, PA_ERR_TIMEOUT);
}

PFN_cuTensorMapEncodeTiled_v12000 g_tc_encode = nullptr;
std::once_flag g_tc_encode_once;

bool tc_encoder() {
  std::call_once(g_tc_encode_once, []() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_tc_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_tc_encode != nullptr;
}

bool tc_encode3(CUtensorMap* map, const void* base, int dtype, const uint64_t (&dims)[3],
                const uint64_t (&strides)[2], const uint32_t (&box)[3]) {
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides[0], strides[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  cuuint32_t es[3] = {1, 1, 1};
  return g_tc_encode(map,
                     dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     3, const_cast<void*>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int D, int G>
cudaError_t launch_tc(const MultiQueryArgs& a, cudaStream_t st) {
  using Ly = TcLayout<D>;
  if (!tc_encoder()) return cudaErrorNotSupported;
  const uint64_t planes = (uint64_t)a.num_blocks * a.num_kv_heads;
  if (planes == 0 || planes > 0x7fffffffull || a.num_tokens <= 0 ||
      a.num_tokens > 0x7fffffffll)
    return cudaErrorInvalidValue;
  const uint32_t R = a.block_size < kTcKv ? (uint32_t)a.block_size : (uint32_t)kTcKv;
  CUtensorMap tq, tk, tv;
  // q [tokens][Hq][D]: a box is one 64-column half of G heads x 128/G tokens
  const bool ok =
      tc_encode3(&tq, a.q, a.dtype, {(uint64_t)D, (uint64_t)a.num_q_heads, (uint64_t)a.num_tokens},
                 {(uint64_t)D * 2, (uint64_t)a.num_q_heads * D * 2},
                 {64u, (uint32_t)G, (uint32_t)(kTcRows / G)}) &&
      // pools [NB][Hkv][B][D] as {D, B, NB*Hkv}: one half of R rows of one slice
      tc_encode3(&tk, a.kc, a.dtype, {(uint64_t)D, (uint64_t)a.block_size, planes},
                 {(uint64_t)D * 2, (uint64_t)a.block_size * D * 2}, {64u, R, 1u}) &&
      tc_encode3(&tv, a.vc, a.dtype, {(uint64_t)D, (uint64_t)a.block_size, planes},
                 {(uint64_t)D * 2, (uint64_t)a.block_size * D * 2}, {64u, R, 1u});
  if (!ok) return cudaErrorInvalidValue;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, []() {
    attr = cudaFuncSetAttribute(multi_query_tc_kernel<T, D, G, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::SMEM);
    if (attr == cudaSuccess)
      attr = cudaFuncSetAttribute(multi_query_tc_kernel<T, D, G, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::SMEM);
  });
  if (attr != cudaSuccess) return attr;
  const int64_t tiles = ((int64_t)a.max_query_len * G + kTcRows - 1) / kTcRows;
  if (tiles == 0 || a.num_seqs == 0) return cudaSuccess;
  if (tiles * a.num_splits > 0x7fffffffll) return cudaErrorInvalidValue;
  dim3 grid((unsigned)(tiles * a.num_splits), a.num_kv_heads, a.num_seqs);
  // runs shorter than one row tile: warps without rows skip their work
  if ((int64_t)a.max_query_len * G < kTcRows)
    multi_query_tc_kernel<T, D, G, true><<<grid, kTcThreads, Ly::SMEM, st>>>(a, tq, tk, tv);
  else
    multi_query_tc_kernel<T, D, G, false><<<grid, kTcThreads, Ly::SMEM, st>>>(a, tq, tk, tv);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_tc_d(const MultiQueryArgs& a, cudaStream_t st) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_tc<T, D, 1>(a, st);
    case 2: return launch_tc<T, D, 2>(a, st);
    case 4: return launch_tc<T, D, 4>(a, st);
    case 8: return launch_tc<T, D, 8>(a, st);
  }
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_tc_t(const MultiQueryArgs& a, cudaStream_t st) {
  if (a.head_size == 64) return launch_tc_d<T, 64>(a, st);
  if (a.head_size == 128) return launch_tc_d<T, 128>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_multi_query_tc(const MultiQueryArgs& a, cudaStream_t st) {
  if (a.dtype == PA_BF16) return launch_tc_t<__nv_bfloat16>(a, st);
  if (a.dtype == PA_F16) return launch_tc_t<__half>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
