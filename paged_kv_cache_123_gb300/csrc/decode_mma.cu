// Paged decode attention on the tensor cores, for query-head groups (GQA).
//
// Same computation as decode_simt.cu ("Visual reading: paged-attention-kv-
// cache", block-wise attention; "vLLM 的 PagedAttention：显存管理如何撑起大模
// 型推理" §2.1: the query heads of a group share one KV head). With a group of
// G query heads per KV head, the per-block work is a dense contraction:
//     S^T[tokens x heads] = K_blk[tokens x D] * Q^T[D x heads]
//     O^T[D x heads]     += V_blk^T[D x tokens] * P^T[tokens x heads]
// so it runs on mma.sync m16n8k16 with the group as the N = 8 side (groups of
// 2 or 4 are zero-padded) and 16 tokens or 16 head dims as the M side.
//
// Work items are (partition, KV head, sequence). Data movement: a producer
// warp walks an item's block table and issues one 4-D tiled TMA load
// (cp.async.bulk.tensor) per block (up to 64 whole token rows, one
// contiguous run in HBM) for K and for V into a ring of 64-token tiles (3
// stages; 4 for fp8 pools), with the 128-byte swizzle so ldmatrix reads hit
// at most two rows per bank group. Four consumer warps take 16 tokens of
// each tile each, keep their own running softmax state (log2 domain), and
// free the stage through an mbarrier; at the end of an item they merge in
// the stage of its last tile and release it afterwards. A CTA takes one
// item, or (MULTI: windowed batches, one wave of CTAs) several in turn, its
// producer running ahead into the next: items blockIdx.x, blockIdx.x +
// gridDim.x, ..., or (the even schedule) an equal share of the batch's
// 64-token tiles: the tiles of all (sequence, KV head) pairs in order, cut
// into gridDim.x consecutive runs, the CTA walking the segments (pieces of
// pairs) of its run; a pair cut between CTAs leaves partial results that
// even_merge_kernel combines. Every wait is bounded: a stuck barrier raises
// an abort flag, the CTA lets its copies in flight land (with its own limit)
// and leaves, and PA_ERR_TIMEOUT is latched.
//
// Rows past the end of the sequence (the tail of the last block, blocks not
// loaded) are masked to -inf in S and zeroed in the V tile before the P*V
// product, so stale or uninitialised pool bytes cannot leak into the output.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "launchers.h"
#include "mma_util.cuh"
#include "tma.cuh"

namespace pa {

constexpr int kMmaConsumers = 4;
constexpr int kMmaThreads = (kMmaConsumers + 1) * 32;
constexpr int kTile = 64;
// stages of the K/V ring: four for fp8 pools (16 KB stages, three CTAs per
// SM: 192 KB in flight per SM, as the 16-bit ring's three 32 KB stages at
// two CTAs per SM), three for 16-bit pools and for one-item CTAs over fp8
// pools with per-block scales, which run four CTAs per SM (more warps to
// cover their dependent scale lookups: 0.67 -> 0.71 of the copy bandwidth
// on the GQA batch; one-scale pools measured no better with four). CTAs
// that walk several items over per-block-scale pools keep three per SM:
// at four (96 registers) their consumers spilled (GQA batch, window 1000:
// 71.8 us against 66.8 us at three).
template <bool KV8, bool SCALED, bool MULTI>
constexpr int ring_stages() { return KV8 ? (SCALED && !MULTI ? 3 : 4) : 3; }
template <bool KV8, bool SCALED, bool MULTI>
constexpr int ctas_per_sm() { return KV8 ? (SCALED && !MULTI ? 4 : 3) : 2; }
// MULTI: an item's query group rides in the stage of its first tile, in a
// slot that keeps the stages 1024-byte aligned (128-byte swizzle), so the
// consumers hold no prefetched query in registers (a one-item CTA loads it
// from global memory while its first tile is in flight instead)
template <typename T, int D, int G, bool MULTI>
constexpr int q_slot_bytes() { return MULTI ? (G * D * (int)sizeof(T) + 1023) / 1024 * 1024 : 0; }
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz
constexpr float kLazyLog2 = 8.f;   // reference maximum moves when exceeded by 2^8
// even schedule: flags of a CTA's record (its last segment): it walked a
// segment, that segment starts at its pair's first tile, ends before its
// last, and is the CTA's only segment
constexpr int kRecNonEmpty = 1, kRecStart0 = 2, kRecCutEnd = 4, kRecSingle = 8;
#define kNegInfM (-__int_as_float(0x7f800000))


// Named barrier 1 over the four consumer warps (128 threads); the _and form
// also returns whether every one of them passed `ok`.
__device__ __forceinline__ void consumers_bar() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}
__device__ __forceinline__ bool consumers_bar_and(bool ok) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n"
      " barrier.cta.red.and.pred po, 1, 128, pi;\n selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(out) : "r"((uint32_t)ok) : "memory");
  return out != 0;
}

// KV8 = the pools hold fp8 (E4M3) codes (head size 128): TMA brings the
// codes (128-byte rows, 128-byte swizzle) and each lane widens the codes it
// needs straight into fp16 mma fragments — K with the head dims of a k-step
// permuted so a lane's codes are contiguous (q uses the same permutation),
// V with two token rows byte-interleaved per head dim — so the products run
// in fp16 without a widened copy in shared memory. k_scale / v_scale are
// the pools' scales (1 for 16-bit pools).
// fp8 pools: half the shared memory per stage and a register budget for
// three CTAs per SM (four with per-block scales), so more warps hide the
// conversion latency.
// MULTI: the CTA walks several items (a.items_per_cta > 1: strided items;
// a.even_ctas > 0: the segments of its even share of the batch's tiles, see
// the top of this file); otherwise it takes work item blockIdx.x.
// SCALED (fp8 pools only): the blocks carry their own scales (a.k_scales /
// a.v_scales [num_blocks][num_kv_heads]). The producer lane that loads a
// block piece also reads its two scales and leaves them beside the stage
// (0 for pieces it does not load). A consumer multiplies each row's logit by
// its K scale, and its softmax weight by the ratio of its V scale to the
// warp's reference, the largest V scale the warp has met so far, before the
// weight is rounded to fp16 for the P*V product: the ratio is at most 1, so
// no weight can overflow, and a weight loses no more than it would with one
// pool-wide scale equal to the reference. When the reference grows the
// warp's output is rescaled with the softmax's own rescale, and the warp's
// output is multiplied by its reference when the warps merge; the
// denominator sums the unscaled weights.
template <typename T, int D, int G, bool KV8, bool MULTI, bool SCALED>
__global__ void __launch_bounds__(kMmaThreads, ctas_per_sm<KV8, SCALED, MULTI>())
decode_mma_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, float k_scale, float v_scale) {
  constexpr int HALVES = D / 64;                 // 128-byte lines per 16-bit token row
  constexpr int ROW_BYTES = HALVES * 128;        // one 16-bit token row (D * 2 bytes)
  constexpr int IN_ROW = KV8 ? D : ROW_BYTES;    // one token row as loaded
  constexpr int KV_BYTES = kTile * IN_ROW;       // K (or V) part of a stage
  constexpr int Q_BYTES = G * D * (int)sizeof(T);
  constexpr int STAGE_BYTES = 2 * KV_BYTES + q_slot_bytes<T, D, G, MULTI>();
  constexpr int PRIV_BYTES = 0;
  constexpr int kSt = ring_stages<KV8, SCALED, MULTI>();
  static_assert(!KV8 || D == 128, "fp8 pools: head size 128 (one 128-byte line per row)");
  // fp8 pools run the products in fp16 whatever the query type: codes widen
  // to fp16 in one conversion. A bf16 query group is first multiplied by the
  // power of two 2^-e that puts its largest magnitude in [2^14, 2^15), which
  // makes the fp16 conversion exact over bf16's whole range (bf16 has 8
  // significant bits, fp16 11; only elements below 2^-28 of the group's
  // largest reach fp16's subnormals), and 2^e goes into the logit scale.
  using MT = typename std::conditional<KV8, __half, T>::type;
  constexpr bool kQRescale = KV8 && std::is_same<T, __nv_bfloat16>::value;
  constexpr int KSTEPS = D / 16;
  static_assert(G == 2 || G == 4 || G == 8 || (KV8 && G == 1), "group");
  static_assert(!SCALED || KV8, "per-block scales: fp8 pools");

  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, reached by pointer arithmetic on the shared
  // array itself so the compiler keeps every access in the shared space
  // (an integer round trip would make them generic loads)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSt * STAGE_BYTES +
                                                kMmaConsumers * PRIV_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kSt);
  // bit p set = piece p of the stage's tile was loaded (written by the
  // producer before it arms the stage's full barrier)
  unsigned* tile_mask = reinterpret_cast<unsigned*>(bars + 2 * kSt) + 1;
  const uint32_t smem0 = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int st) { return bar0 + 8u * st; };
  auto empty_bar = [&](int st) { return bar0 + 8u * (kSt + st); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;
  const int B = a.block_size;
  const int bshift = __ffs(B) - 1;
  const int R = B < kTile ? B : kTile;           // rows per TMA box
  // work items (partition, KV head, sequence), partition fastest
  const int n_items = a.num_splits * Hkv * a.num_seqs;
  const bool even = MULTI && a.even_ctas > 0;   // the even schedule
  // per-warp row maxima and sums for the merge of an item ([4][8] each)
  float* sm_m = reinterpret_cast<float*>(tile_mask + kSt);
  float* sm_l = sm_m + kMmaConsumers * 8;
  // SCALED: per stage, each piece's K and V scale ([kSt][8] each), and the
  // item's largest V scale up to that tile ([kSt])
  float* st_ks = sm_l + kMmaConsumers * 8;
  float* st_vs = st_ks + kSt * 8;
  float* st_vref = st_vs + kSt * 8;
  // even schedule: the start of this CTA's share, found by all threads
  // (per-warp sums [5], tiles g0 and g1 of the batch, the offset of g0 in its
  // sequence's tiles; the sequence and its length)
  long long* ev_ll = reinterpret_cast<long long*>(
      smem + ((reinterpret_cast<uint8_t*>(st_vref + kSt) - smem + 7) & ~7));
  int* ev_i = reinterpret_cast<int*>(ev_ll + 8);
  struct Item {
    int s, kvh, split, L, lo, t0, t1, ntiles;
    bool bad, zero_out;
    bool complete;        // covers the pair's whole range: the output is final
    bool first;           // even: the CTA's first segment (partial slot 0, else 1)
    bool start0, cut_end; // even: starts at the pair's first tile / ends before its last
  };
  auto bad_len = [&](int L) {
    return L < 0 || L > a.max_seq_len || (int64_t)L > a.table_stride * a.block_size;
  };
  auto item_at = [&](int idx) {
    Item im;
    im.split = idx % a.num_splits;
    const int rest = idx / a.num_splits;
    im.kvh = rest % Hkv;
    im.s = rest / Hkv;
    im.L = a.seq_lens[im.s];
    im.bad = bad_len(im.L);
    // an empty or invalid sequence: its first partition writes zeros
    im.zero_out = (im.bad || im.L == 0) && im.split == 0;
    im.lo = 0; im.t0 = 0; im.t1 = 0; im.ntiles = 0;
    im.complete = true; im.first = true; im.start0 = true; im.cut_end = false;
    if (!im.bad && im.L > 0) {
      im.lo = window_lo(im.L, a.window);
      im.t0 = window_base(im.lo) + im.split * a.partition;
      if (im.t0 < im.L) {
        im.t1 = min(im.L, im.t0 + a.partition);
        im.complete = (im.L - window_base(im.lo) + a.partition - 1) / a.partition == 1;
        im.ntiles = (im.t1 - im.t0 + kTile - 1) / kTile;
      }
    }
    return im;
  };
  // even schedule: tiles of a sequence of length L (0 for empty or invalid lengths,
  // whose zeros even_merge_kernel writes)
  auto seq_tiles = [&](int L) -> int {
    if (L <= 0 || bad_len(L)) return 0;
    return (L - window_base(window_lo(L, a.window)) + kTile - 1) / kTile;
  };
  auto len_of = [&](int s) { return s < a.num_seqs ? a.seq_lens[s] : 0; };
  // even schedule: cursor over this CTA's share: g = the batch's next tile (pair
  // s * Hkv + kvh, tile ta of the pair's ntl), g1 = the end of the share;
  // Ln = the next sequence's length, loaded ahead
  struct Cursor {
    long long g, g1;
    int s, kvh, ta, L, ntl, Ln;
    bool first;
  };
  auto cursor_item = [&](const Cursor& c) {
    Item im;
    im.s = c.s; im.kvh = c.kvh; im.split = 0; im.L = c.L;
    im.bad = false; im.zero_out = false;
    im.lo = window_lo(c.L, a.window);
    const int base = window_base(im.lo);
    const int tb = (int)min((long long)c.ntl, c.ta + (c.g1 - c.g));
    im.t0 = base + c.ta * kTile;
    im.t1 = min(c.L, base + tb * kTile);
    im.ntiles = tb - c.ta;
    im.first = c.first;
    im.start0 = c.ta == 0;
    im.cut_end = tb < c.ntl;
    im.complete = im.start0 && !im.cut_end;
    return im;
  };
  auto cursor_next = [&](Cursor& c) {
    c.g += (int)min((long long)c.ntl, c.ta + (c.g1 - c.g)) - c.ta;
    c.ta = 0;
    c.first = false;
    if (c.g >= c.g1 || ++c.kvh < Hkv) return;
    c.kvh = 0;
    do {                                   // the next sequence with tiles
      if (c.s + 1 >= a.num_seqs) {         // (none: lengths inconsistent, stop)
        c.g = c.g1;
        return;
      }
      ++c.s;
      c.L = c.Ln;
      c.Ln = len_of(c.s + 1);
      c.ntl = seq_tiles(c.L);
    } while (c.ntl == 0);
  };
  // the CTA's items: item blockIdx.x, items blockIdx.x + k * gridDim.x
  // (MULTI), or the segments of its even share
  struct Iter {
    Cursor c;
    int idx;
    bool done;
  };
  auto iter_begin = [&]() {
    Iter w;
    w.idx = blockIdx.x;
    if (even) {
      w.c.g = ev_ll[5];
      w.c.g1 = ev_ll[6];
      w.done = ev_i[0] < 0 || w.c.g >= w.c.g1;
      if (!w.done) {
        w.c.s = ev_i[0];
        w.c.L = ev_i[1];
        w.c.ntl = seq_tiles(w.c.L);
        const long long off = ev_ll[7];
        w.c.kvh = (int)(off / w.c.ntl);
        w.c.ta = (int)(off - (long long)w.c.kvh * w.c.ntl);
        w.c.Ln = len_of(w.c.s + 1);
        w.c.first = true;
      }
    } else {
      w.done = w.idx >= n_items;
    }
    return w;
  };
  auto iter_item = [&](const Iter& w) { return even ? cursor_item(w.c) : item_at(w.idx); };
  auto iter_next = [&](Iter& w) {
    if (even) {
      cursor_next(w.c);
      w.done = w.c.g >= w.c.g1;
    } else if (MULTI) {
      w.idx += gridDim.x;
      w.done = w.idx >= n_items;
    } else {
      w.done = true;
    }
  };

  if (threadIdx.x == 0) {
    for (int st = 0; st < kSt; ++st) {
      mbar_init(full_bar(st), 1);
      mbar_init(empty_bar(st), kMmaConsumers);
    }
    *abort_flag = 0;
    if (even) ev_i[0] = -1;
    mbar_fence_init();
  }
  griddep_wait();
  if (even) {
    // the batch's tiles T (every thread sums a contiguous range of
    // sequences, then an exclusive scan over the threads); this CTA's share
    // is tiles [g0, g1) with g0 = floor(blockIdx.x * T / gridDim.x), and
    // the thread whose sequences hold tile g0 finds its sequence
    const int S = a.num_seqs;
    const int K = (S + kMmaThreads - 1) / kMmaThreads;
    const int sb = threadIdx.x * K;
    long long mine = 0;
    for (int j = 0; j < K; ++j)
      if (sb + j < S) mine += seq_tiles(a.seq_lens[sb + j]);
    long long inc = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += v;
    }
    if (lane == 31) ev_ll[warp] = inc;
    __syncthreads();
    long long before = 0, total = 0;
#pragma unroll
    for (int w = 0; w <= kMmaConsumers; ++w) {
      const long long t = ev_ll[w];
      if (w < warp) before += t;
      total += t;
    }
    const long long tiles = total * Hkv, C = gridDim.x;
    const long long g0 = (long long)blockIdx.x * tiles / C;
    const long long g1 = ((long long)blockIdx.x + 1) * tiles / C;
    long long cum = (before + inc - mine) * Hkv;
    if (g0 < g1 && cum <= g0 && g0 < cum + mine * Hkv) {
      for (int j = 0; j < K && sb + j < S; ++j) {
        const int L = a.seq_lens[sb + j];
        const long long t = (long long)seq_tiles(L) * Hkv;
        if (g0 < cum + t) {
          ev_i[0] = sb + j;
          ev_i[1] = L;
          ev_ll[7] = g0 - cum;
          break;
        }
        cum += t;
      }
    }
    __syncthreads();        // every thread has read the warp sums
    if (threadIdx.x == 0) {
      ev_ll[5] = g0;
      ev_ll[6] = g1;
    }
  }
  __syncthreads();
  // the next launch (the combine or merge) may be scheduled now; it waits
  // for this grid to complete before it reads the partials
  griddep_launch();

  if (warp == kMmaConsumers) {
    // ---------------- producer warp: lane p owns piece p (R rows of one
    // block) of each tile; the table entries of a tile are read in parallel
    // before waiting for the stage, and each lane issues its own TMA loads.
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
    }
    const int npieces = kTile / R;             // <= 8 (R >= 8)
    int it = 0;                                // tiles issued so far: the ring position
    bool run = true;
    auto in_pool = [&](int64_t b) { return b >= 0 && b < a.num_blocks; };
    // Issue the tile starting at token ts of KV head kvh into the next
    // stage: lane p loads piece p (R rows of block blk) when `need`; the
    // first tile of an item (qs = its sequence, else -1) also brings the
    // item's query group. SCALED: ksv and rsv are the piece's K and V
    // scales, vrt the largest V scale of the item so far (the reference the
    // consumers' output is kept in).
    auto issue_tile = [&](int ts, int kvh, int64_t blk, bool need, float ksv, float rsv,
                          float vrt, int qs) -> bool {
      const int st = it % kSt;
      const int tok = ts + lane * R;
      const bool mine = need && in_pool(blk);
      if (need && !mine) latch(a.err, PA_ERR_OUT_OF_RANGE);
      const unsigned pm = __ballot_sync(0xffffffffu, mine);
      int ok = 1;
      if constexpr (SCALED) {
        if (lane == 0 && it >= kSt)
          ok = mbar_wait_bounded(empty_bar(st), ((it / kSt) - 1) & 1, abort_flag, kWaitCycles);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return false;
        if (lane < npieces) {
          st_ks[st * 8 + lane] = ksv;
          st_vs[st * 8 + lane] = rsv;
        }
        // the warp's scale stores come before lane 0's arrive (release), and
        // the arrive before any lane's copy
        __syncwarp();
        if (lane == 0) {
          st_vref[st] = vrt;
          tile_mask[st] = pm;
          mbar_arrive_expect_tx(full_bar(st), (uint32_t)__popc(pm) * 2u * R * IN_ROW +
                                                  (qs >= 0 ? (uint32_t)Q_BYTES : 0u));
        }
        __syncwarp();
      } else {
        if (lane == 0) {
          if (it >= kSt)
            ok = mbar_wait_bounded(empty_bar(st), ((it / kSt) - 1) & 1, abort_flag, kWaitCycles);
          if (ok) {
            tile_mask[st] = pm;
            mbar_arrive_expect_tx(full_bar(st), (uint32_t)__popc(pm) * 2u * R * IN_ROW +
                                                    (qs >= 0 ? (uint32_t)Q_BYTES : 0u));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return false;
      }
      if (lane == 0 && qs >= 0)
        bulk_load(smem0 + st * STAGE_BYTES + 2 * KV_BYTES,
                  reinterpret_cast<const T*>(a.q) + ((int64_t)qs * Hq + (int64_t)kvh * G) * D,
                  (uint32_t)Q_BYTES, full_bar(st));
      if (mine) {
        const uint32_t kdst = smem0 + st * STAGE_BYTES + lane * R * IN_ROW;
        const uint32_t vdst = kdst + KV_BYTES;
        const int z = (int)(blk * Hkv + kvh);
        const int y = tok & (B - 1);
        if (KV8) {
          tma_load_3d(kdst, &tmK, 0, y, z, full_bar(st));
          tma_load_3d(vdst, &tmV, 0, y, z, full_bar(st));
        } else {
          tma_load_4d(kdst, &tmK, 0, 0, y, z, full_bar(st));
          tma_load_4d(vdst, &tmV, 0, 0, y, z, full_bar(st));
        }
      }
      ++it;
      return true;
    };
    if constexpr (!SCALED) {
      // the table entries of a tile are read in parallel (one lane per
      // piece) right before its stage is awaited
      for (Iter w = iter_begin(); run && !w.done; iter_next(w)) {
        const Item im = iter_item(w);
        const int32_t* trow = a.tables + (int64_t)im.s * a.table_stride;
        for (int i = 0; i < im.ntiles; ++i) {
          const int ts = im.t0 + i * kTile;
          const int tok = ts + lane * R;
          const bool need = lane < npieces && tok < min(im.t1, ts + kTile) && tok + R > im.lo;
          const int64_t blk = need ? (int64_t)trow[tok >> bshift] : -1;
          if (!issue_tile(ts, im.kvh, blk, need, 0.f, 0.f, 0.f, MULTI && i == 0 ? im.s : -1)) {
            run = false;
            break;
          }
        }
      }
    } else {
      // per-block scales: each piece's scales are read through its table
      // entry, two dependent loads. They run ahead of the copies in a
      // software pipeline over the CTA's tiles: while tile k is issued, the
      // table entries of tile k+2 and the scales of tile k+1 are in flight.
      // One cursor (gw, gim, gi) walks the items; the pipeline holds only
      // small per-tile descriptors.
      struct TD {
        int s, kvh, ts;
        bool need, first;     // this lane's piece is attended; the item's first tile
      };
      Iter gw = iter_begin();
      Item gim;
      int gi = 0;
      if (!gw.done) gim = iter_item(gw);
      auto settle = [&]() {                    // skip items without tiles
        while (!gw.done && gi >= gim.ntiles) {
          iter_next(gw);
          gi = 0;
          if (!gw.done) gim = iter_item(gw);
        }
      };
      settle();
      // the next tile's descriptor (valid = false past the last tile)
      auto gen = [&](TD& td) -> bool {
        if (gw.done) {
          td.need = false;
          td.first = false;
          return false;
        }
        td.s = gim.s;
        td.kvh = gim.kvh;
        td.ts = gim.t0 + gi * kTile;
        td.first = gi == 0;
        const int tok = td.ts + lane * R;
        td.need = lane < npieces && tok < min(gim.t1, td.ts + kTile) && tok + R > gim.lo;
        ++gi;
        settle();
        return true;
      };
      auto table_of = [&](const TD& td) -> int64_t {
        if (!td.need) return -1;
        return a.tables[(int64_t)td.s * a.table_stride + ((td.ts + lane * R) >> bshift)];
      };
      TD d0, d1, d2;
      bool v0 = gen(d0), v1 = gen(d1);
      int64_t b0 = table_of(d0), b1 = table_of(d1);
      // pieces that are not loaded get scales 0 (their rows are masked)
      float ks0 = 0.f, vs0 = 0.f, vrun = 0.f;
      if (in_pool(b0)) {
        ks0 = a.k_scales[b0 * Hkv + d0.kvh];
        vs0 = a.v_scales[b0 * Hkv + d0.kvh];
      }
      while (run && v0) {
        const bool v2 = gen(d2);
        const int64_t b2 = table_of(d2);       // two tiles ahead
        float ks1 = 0.f, vs1 = 0.f;
        if (in_pool(b1)) {                     // one tile ahead
          ks1 = a.k_scales[b1 * Hkv + d1.kvh];
          vs1 = a.v_scales[b1 * Hkv + d1.kvh];
        }
        // the item's running maximum V scale (scales are >= 0, so their
        // bit patterns order like the values)
        if (d0.first) vrun = 0.f;
        vrun = fmaxf(vrun, __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(vs0))));
        if (!issue_tile(d0.ts, d0.kvh, b0, d0.need, ks0, vs0, vrun,
                        MULTI && d0.first ? d0.s : -1)) {
          run = false;
          break;
        }
        d0 = d1;
        d1 = d2;
        v0 = v1;
        v1 = v2;
        b0 = b1;
        b1 = b2;
        ks0 = ks1;
        vs0 = vs1;
      }
    }
    // let the loads this CTA issued land before it can leave (also after a
    // timeout: this wait has its own limit and ignores the abort flag)
    if (lane == 0)
      for (int j = it > kSt ? it - kSt : 0; j < it; ++j)
        mbar_wait_drain(full_bar(j % kSt), (j / kSt) & 1, kWaitCycles);
  } else {
    // ---------------- consumers
    const int n = lane >> 2, c = lane & 3;
    // pieces (R rows of one block) of this lane's rows n and n+8 of the
    // warp's 16 in every tile (R is a power of two)
    const int rshift = __ffs(R) - 1;
    const int pA = (warp * 16 + n) >> rshift, pB = (warp * 16 + n + 8) >> rshift;
    const float sl2 = a.scale * kLog2e * k_scale;
    T* out = reinterpret_cast<T*>(a.out);
    int it = 0;                                // tiles consumed so far: the ring position
    bool run = true;
    // query fragments of an item from its query group [G][D] (q_read: in
    // the slot of the item's first stage, or in global memory), then in the
    // products' type with the factor qmul by which the products must be
    // multiplied (q_finish)
    auto q_read = [&](const T* qb, uint32_t (&qd)[KSTEPS][2]) {
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        if (n < G) {
          // fp8 pools: k-step ks, lane quad c covers head dims
          // c*D/4 + 4ks .. +3 (a fixed permutation of the contraction order,
          // applied to K the same way) so a lane's codes are contiguous
          const int d0 = KV8 ? c * (D / 4) + ks * 4 : ks * 16 + 2 * c;
          const int d1 = KV8 ? d0 + 2 : d0 + 8;
          qd[ks][0] = *reinterpret_cast<const uint32_t*>(qb + n * D + d0);
          qd[ks][1] = *reinterpret_cast<const uint32_t*>(qb + n * D + d1);
        } else {
          qd[ks][0] = qd[ks][1] = 0u;
        }
      }
    };
    auto q_finish = [&](uint32_t (&qd)[KSTEPS][2], float& qmul) {
      qmul = 1.f;
      if constexpr (kQRescale) {
        // the lanes of the warp hold the whole group between them
        float mx = 0.f;
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float2 f = MmaOps<T>::unpack(qd[ks][j]);
            mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        // e = floor(log2(mx)) - 14, kept >= -126 so 2^e and 2^-e are normal
        // fp32 values (a group below 2^-112 only loses digits it cannot use)
        const int e = mx > 0.f ? max(((__float_as_int(mx) >> 23) & 0xff) - 127 - 14, -126) : 0;
        const float down = __int_as_float((127 - e) << 23);
        qmul = __int_as_float((127 + e) << 23);
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float2 f = MmaOps<T>::unpack(qd[ks][j]);
            qd[ks][j] = MmaOps<MT>::pack(f.x * down, f.y * down);
          }
      } else {
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks)
#pragma unroll
          for (int j = 0; j < 2; ++j) qd[ks][j] = to_mma_pair<T, MT>(qd[ks][j]);
      }
    };
    Iter cw = iter_begin();
    // even schedule: the segments walked and the last one (for the merge
    // launch)
    int nseg = 0;
    int last_pair = 0;
    bool last_start0 = false, last_cut_end = false;
    while (run && !cw.done) {
    const Item im = iter_item(cw);
    iter_next(cw);
    uint32_t qf[KSTEPS][2];
    float qmul = 1.f;
    if (im.zero_out) {
      if (im.L != 0 && threadIdx.x == 0) latch(a.err, PA_ERR_OUT_OF_RANGE);
      for (int i = threadIdx.x; i < G * D; i += kMmaConsumers * 32)
        out[((int64_t)im.s * Hq + (int64_t)im.kvh * G) * D + i] = Vec<T>::cvt_out(0.f);
      continue;
    }
    if (im.ntiles == 0) continue;
    const int s = im.s, kvh = im.kvh, split = im.split, lo = im.lo;
    const int t0 = im.t0, t1 = im.t1, ntiles = im.ntiles;
    ++nseg;
    last_pair = s * Hkv + kvh;
    last_start0 = im.start0;
    last_cut_end = im.cut_end;
    // merge state, per consumer warp; heads 2c and 2c+1 of this lane
    float m0 = kNegInfM, m1 = kNegInfM, l0 = 0.f, l1 = 0.f;
    float o[KSTEPS][4];
#pragma unroll
    for (int i = 0; i < KSTEPS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float sl2q = sl2;
    if (!MULTI) {
      q_read(reinterpret_cast<const T*>(a.q) + ((int64_t)s * Hq + (int64_t)kvh * G) * D, qf);
      q_finish(qf, qmul);
      sl2q = sl2 * qmul;
    }
    // SCALED: the reference V scale the warp's output is kept in (0 until
    // the first tile) and its reciprocal
    float vref = 0.f, inv_vref = 0.f;
    bool ok = true;
    for (int i = 0; i < ntiles; ++i, ++it) {
      const int st = it % kSt;
      // the stage of an item's last tile is released after the merge, which
      // uses it
      const bool last = i + 1 == ntiles;
      if (!mbar_wait_bounded(full_bar(st), (it / kSt) & 1, abort_flag, kWaitCycles)) {
        ok = false;
        break;
      }
      if (MULTI && i == 0) {     // the item's query group came with its first tile
        q_read(reinterpret_cast<const T*>(smem + st * STAGE_BYTES + 2 * KV_BYTES), qf);
        q_finish(qf, qmul);
        sl2q = sl2 * qmul;
      }
      const int ts = t0 + i * kTile;
      const int te = min(t1, ts + kTile);
      const int r0 = ts + warp * 16;   // first token of this warp's 16 rows
      const uint32_t kst = smem0 + st * STAGE_BYTES;
      const uint32_t vst = kst + KV_BYTES;
      if (r0 < te) {
        bool row_ok = false;
        {
          const int r = warp * 16 + (lane & 15);   // row inside the tile
          row_ok = (ts + r < te) && (ts + r >= lo) && ((tile_mask[st] >> (r / R)) & 1u);
        }
        const unsigned okm = __ballot_sync(0xffffffffu, row_ok) & 0xffffu;
        const uint32_t kb = kst, vb = vst;
        const int rbase = warp * 16;
        if (!KV8 && okm != 0xffffu) {
          const int r = lane & 15, h = lane >> 4;
          if (h < HALVES && !((okm >> r) & 1u)) {
            uint4* p = reinterpret_cast<uint4*>(smem + (vst - smem0) +
                                                (warp * 16 + r) * ROW_BYTES + h * 128);
#pragma unroll
            for (int j = 0; j < 8; ++j) p[j] = make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
        }
        // S^T = K * Q^T for this warp's 16 tokens
        float sacc[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (KV8) {
          // codes of rows n and n+8, head dims c*D/4 .. +D/4-1 (two 16-byte
          // chunks, 128-byte swizzle), widened straight into A fragments
          const uint8_t* kbase = smem + (kst - smem0);
          const int ra = warp * 16 + n, rb = ra + 8;
          uint4 ka[2], kq[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            ka[h] = *reinterpret_cast<const uint4*>(kbase + ra * 128 + (((2 * c + h) ^ (ra & 7)) << 4));
            kq[h] = *reinterpret_cast<const uint4*>(kbase + rb * 128 + (((2 * c + h) ^ (rb & 7)) << 4));
          }
          const uint32_t wa[8] = {ka[0].x, ka[0].y, ka[0].z, ka[0].w, ka[1].x, ka[1].y, ka[1].z, ka[1].w};
          const uint32_t wb[8] = {kq[0].x, kq[0].y, kq[0].z, kq[0].w, kq[1].x, kq[1].y, kq[1].z, kq[1].w};
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            uint32_t af[4];
            e4m3x4_to_f16x2x2(wa[ks], af[0], af[2]);
            e4m3x4_to_f16x2x2(wb[ks], af[1], af[3]);
            MmaOps<MT>::mma(sacc, af, qf[ks][0], qf[ks][1]);
          }
        } else {
          const int j = lane >> 3;
          const int row = rbase + (j & 1) * 8 + (lane & 7);
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            const int dch = ks * 2 + (j >> 1);
            uint32_t af[4];
            ldsm_x4(af, swz<HALVES>(kb, row, dch));
            MmaOps<MT>::mma(sacc, af, qf[ks][0], qf[ks][1]);
          }
        }
        const bool okA = (okm >> n) & 1u, okB = (okm >> (n + 8)) & 1u;
        // SCALED: rows n and n+8 take the K scales of their pieces and
        // their V scales relative to the reference; when the reference grew,
        // the output so far is rescaled to it
        float slA = sl2q, slB = sl2q, rA = 0.f, rB = 0.f, cv = 1.f;
        if constexpr (SCALED) {
          const float vr = st_vref[st];
          if (vr != vref) {              // warp-uniform; vr > vref here
            cv = vref / vr;              // 0 the first time: nothing to rescale
            vref = vr;
            inv_vref = 1.f / vr;
          }
          slA *= st_ks[st * 8 + pA];
          slB *= st_ks[st * 8 + pB];
          rA = st_vs[st * 8 + pA] * inv_vref;
          rB = st_vs[st * 8 + pB] * inv_vref;
        }
        const float x0 = okA ? sacc[0] * slA : kNegInfM;   // row n,   head 2c
        const float x1 = okA ? sacc[1] * slA : kNegInfM;   // row n,   head 2c+1
        const float x2 = okB ? sacc[2] * slB : kNegInfM;   // row n+8, head 2c
        const float x3 = okB ? sacc[3] * slB : kNegInfM;   // row n+8, head 2c+1
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        // fp8 pools (ALU-bound): lazy reference: a head's reference maximum
        // m moves (to the tile's maximum) only when the tile's maximum
        // exceeds it by more than 2^kLazyLog2, so the weights 2^(x - m) stay
        // below 2^8 (exact in fp16 as far as its rounding goes) and the
        // output and sums are rescaled only on those rare tiles, in a
        // warp-uniform branch; the final division and the merges use the
        // same reference (GQA batch 216 -> 211 us, Llama-7B 95.6 -> 92.8 us).
        // 16-bit pools (HBM-bound) keep the exact maximum and rescale every
        // tile (the lazy form measured 0.6 % slower there).
        const float lazy = KV8 ? kLazyLog2 : 0.f;
        const bool up0 = mx0 > m0 + lazy, up1 = mx1 > m1 + lazy;
        float al0 = 1.f, al1 = 1.f;
        bool rescale = !KV8 || (SCALED && cv != 1.f);
        if (!KV8 || __any_sync(0xffffffffu, up0 || up1)) {
          if (up0) {
            al0 = exp2f(m0 - mx0);       // 0 on the first tile (m0 = -inf)
            m0 = mx0;
          }
          if (up1) {
            al1 = exp2f(m1 - mx1);
            m1 = mx1;
          }
          rescale = true;
        }
        const bool live0 = m0 != kNegInfM, live1 = m1 != kNegInfM;
        const float p0 = live0 ? exp2f(x0 - m0) : 0.f;
        const float p2 = live0 ? exp2f(x2 - m0) : 0.f;
        const float p1 = live1 ? exp2f(x1 - m1) : 0.f;
        const float p3 = live1 ? exp2f(x3 - m1) : 0.f;
        uint32_t cA, cB;
        float aO0 = al0, aO1 = al1;      // rescale of the output
        if constexpr (SCALED) {
          cA = MmaOps<MT>::pack(p0 * rA, p1 * rA);     // rA, rB <= 1
          cB = MmaOps<MT>::pack(p2 * rB, p3 * rB);
          l0 = l0 * al0 + p0 + p2;
          l1 = l1 * al1 + p1 + p3;
          aO0 *= cv;
          aO1 *= cv;
        } else {
          cA = MmaOps<MT>::pack(p0, p1);
          cB = MmaOps<MT>::pack(p2, p3);
          // the denominator sums the same rounded weights the MMA multiplies
          const float2 fA = MmaOps<MT>::unpack(cA), fB = MmaOps<MT>::unpack(cB);
          l0 = l0 * al0 + fA.x + fB.x;
          l1 = l1 * al1 + fA.y + fB.y;
        }
        if (rescale) {
#pragma unroll
          for (int mt = 0; mt < KSTEPS; ++mt) {
            o[mt][0] *= aO0; o[mt][1] *= aO1; o[mt][2] *= aO0; o[mt][3] *= aO1;
          }
        }
        const uint32_t pb0 = movmatrix_trans(cA);
        const uint32_t pb1 = movmatrix_trans(cB);
        // O^T += V^T * P^T
        if constexpr (KV8) {
          // token rows 2c, 2c+1, 2c+8, 2c+9, head dims n*16 .. +15 (one
          // 16-byte chunk each); bytes of rows paired per head dim; the M
          // order of this product is head dim n*16 + 8*(row >= 8) + mt
          const uint8_t* vbase = smem + (vst - smem0);
          uint32_t w[4][4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int row = warp * 16 + 2 * c + (r & 1) + (r >> 1) * 8;
            const uint4 v = *reinterpret_cast<const uint4*>(vbase + row * 128 + ((n ^ (row & 7)) << 4));
            w[r][0] = v.x; w[r][1] = v.y; w[r][2] = v.z; w[r][3] = v.w;
          }
          if (okm != 0xffffu) {   // warp-uniform: only partial tiles pay the masking
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              if (!((okm >> (2 * c + (r & 1) + (r >> 1) * 8)) & 1u))
                w[r][0] = w[r][1] = w[r][2] = w[r][3] = 0u;
            }
          }
          // (token pair, head dim j) as f16x2, widened half the words at a
          // time next to the four products that use them (m-tiles 4h..4h+3
          // take code words h and h+2), so fewer widened values are live
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t p01[2][4], p23[2][4];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int q4 = hh + 2 * k;
              const uint32_t lo01 = __byte_perm(w[0][q4], w[1][q4], 0x5140);
              const uint32_t hi01 = __byte_perm(w[0][q4], w[1][q4], 0x7362);
              const uint32_t lo23 = __byte_perm(w[2][q4], w[3][q4], 0x5140);
              const uint32_t hi23 = __byte_perm(w[2][q4], w[3][q4], 0x7362);
              e4m3x4_to_f16x2x2(lo01, p01[k][0], p01[k][1]);
              e4m3x4_to_f16x2x2(hi01, p01[k][2], p01[k][3]);
              e4m3x4_to_f16x2x2(lo23, p23[k][0], p23[k][1]);
              e4m3x4_to_f16x2x2(hi23, p23[k][2], p23[k][3]);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t af[4] = {p01[0][j], p01[1][j], p23[0][j], p23[1][j]};
              MmaOps<MT>::mma(o[4 * hh + j], af, pb0, pb1);
            }
          }
        } else {
          const int j = lane >> 3;
          const int row = rbase + (j >> 1) * 8 + (lane & 7);
#pragma unroll
          for (int mt = 0; mt < KSTEPS; ++mt) {
            const int dch = mt * 2 + (j & 1);
            uint32_t af[4];
            ldsm_x4_trans(af, swz<HALVES>(vb, row, dch));
            MmaOps<MT>::mma(o[mt], af, pb0, pb1);
          }
        }
        if (!KV8 && okm != 0xffffu) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && !last) mbar_arrive(empty_bar(st));
      } else {
        __syncwarp();
        if (lane == 0 && !last) mbar_arrive(empty_bar(st));
      }
    }
    // the four warps agree that every tile of the item arrived (a timed-out
    // wait anywhere stops the CTA; every warp gets here either way) and
    // that all of them have read the last tile's stage
    if (!consumers_bar_and(ok)) {
      run = false;
      break;
    }
    // sum the per-lane denominators over the 8 lanes that share a head pair
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    // merge the four consumer warps in the stage of the item's last tile
    // (16 KB of fp32 partial outputs; maxima and sums beside the barriers)
    const int st_last = (it - 1) % kSt;
    float* sm_o = reinterpret_cast<float*>(smem + st_last * STAGE_BYTES);   // [4][8][D]
    const float ovs = SCALED ? vref : 1.f;
    {
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) {
      float* base = sm_o + warp * 8 * D;
      // head dim of M rows n and n+8 of m-tile mt
      const int da = KV8 ? n * 16 + mt : mt * 16 + n;
      const int db = KV8 ? n * 16 + 8 + mt : mt * 16 + n + 8;
      // SCALED: back to the values' own units (vref is 1 otherwise)
      base[(2 * c) * D + da] = o[mt][0] * ovs;
      base[(2 * c + 1) * D + da] = o[mt][1] * ovs;
      base[(2 * c) * D + db] = o[mt][2] * ovs;
      base[(2 * c + 1) * D + db] = o[mt][3] * ovs;
    }
    if (n == 0) {
      sm_m[warp * 8 + 2 * c] = m0;
      sm_m[warp * 8 + 2 * c + 1] = m1;
      sm_l[warp * 8 + 2 * c] = l0;
      sm_l[warp * 8 + 2 * c + 1] = l1;
    }
    }
    consumers_bar();
    // per head g (thread g): the warps' weights 2^(m_w - M) (times v_scale)
    // replace their maxima in sm_m; sm_l keeps 1 / sum (column g of warp 0),
    // M (warp 1) and the sum (warp 2)
    if (threadIdx.x < G) {
      const int g = threadIdx.x;
      float M = kNegInfM;
#pragma unroll
      for (int w = 0; w < kMmaConsumers; ++w) M = fmaxf(M, sm_m[w * 8 + g]);
      float Ls = 0.f;
#pragma unroll
      for (int w = 0; w < kMmaConsumers; ++w) {
        const float mw = sm_m[w * 8 + g];
        const float wt = (mw == kNegInfM) ? 0.f : exp2f(mw - M);
        Ls += sm_l[w * 8 + g] * wt;
        sm_m[w * 8 + g] = wt * v_scale;
      }
      sm_l[g] = Ls > 0.f ? 1.f / Ls : 0.f;
      sm_l[8 + g] = M;
      sm_l[16 + g] = Ls;
    }
    consumers_bar();
    for (int e = threadIdx.x; e < G * D; e += kMmaConsumers * 32) {
    const int g = e / D, d = e - g * D;
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < kMmaConsumers; ++w) O += sm_o[(w * 8 + g) * D + d] * sm_m[w * 8 + g];
    const float M = sm_l[8 + g], Ls = sm_l[16 + g];
    const int h = kvh * G + g;
    if (im.complete) {
      out[((int64_t)s * Hq + h) * D + d] = Vec<T>::cvt_out(O * sm_l[g]);
    } else if (even) {
      // a pair cut between CTAs: the CTA's first segment in slot 0, its
      // last in slot 1
      const int64_t slot = ((int64_t)blockIdx.x * 2 + (im.first ? 0 : 1)) * G + g;
      a.ws_acc[slot * D + d] = O;
      if (d == 0) { a.ws_ml[2 * slot] = M; a.ws_ml[2 * slot + 1] = Ls; }
    } else {
      const int64_t slot = ((int64_t)s * Hq + h) * a.num_splits + split;
      a.ws_acc[slot * D + d] = O;
      if (d == 0) { a.ws_ml[2 * slot] = M; a.ws_ml[2 * slot + 1] = Ls; }
    }
    }
    // the merge area has been read: the stage may be refilled by TMA
    consumers_bar();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(st_last));
    }
    // even schedule: the record even_merge_kernel reads: the pair of the
    // CTA's last segment and how it was cut (nothing, after a timeout)
    if (even && threadIdx.x == 0) {
      int flags = 0;
      if (run && nseg > 0)
        flags = kRecNonEmpty | (last_start0 ? kRecStart0 : 0) | (last_cut_end ? kRecCutEnd : 0) |
                (nseg == 1 ? kRecSingle : 0);
      a.ws_rec[2 * blockIdx.x] = last_pair;
      a.ws_rec[2 * blockIdx.x + 1] = flags;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) latch(a.err, PA_ERR_TIMEOUT);
}

// The second launch of an even-schedule call, one CTA of kMergeThreads threads per
// CTA of the attention launch (c = blockIdx.x, C = gridDim.x):
//  - sequences s = c, c + C, ... that are empty or invalid get zero outputs
//    (invalid ones also latch PA_ERR_OUT_OF_RANGE): they have no tiles, so
//    no attention CTA visits them, and this runs before the attention
//    launch has finished (programmatic dependent launch);
//  - if attention CTA c holds the start of a pair that continues into the
//    following CTAs (its last segment starts at the pair's first tile and
//    ends before its last), this CTA merges the pair's partial results:
//    CTA c's (slot 0 if that segment was its only one, else slot 1), then
//    slot 0 of every following CTA with a segment up to the one where the
//    pair ends, with the log-sum-exp weights of combine_kernel:
//        M = max_p m_p,  w_p = 2^(m_p - M),  o = sum_p w_p acc_p / sum_p w_p l_p
// Warp 0 reads this CTA's record and the following ones 32 at a time and
// lists the pieces in shared memory; each thread then merges its output
// elements four pieces at a time (online: a running maximum with rescale),
// with all loads of a step independent of each other.
constexpr int kMergeThreads = 256;
template <typename T, int D, int G>
__global__ void __launch_bounds__(kMergeThreads) even_merge_kernel(const DecodeArgs a) {
  extern __shared__ int pieces[];          // [gridDim.x]: partial-slot indices k*2+slot
  __shared__ int n_pieces, head_pair;
  const int c = blockIdx.x, C = gridDim.x;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;
  T* out = reinterpret_cast<T*>(a.out);
  for (int s = c; s < a.num_seqs; s += C) {
    const int L = a.seq_lens[s];
    const bool bad = L < 0 || L > a.max_seq_len || (int64_t)L > a.table_stride * a.block_size;
    if (bad || L == 0) {
      if (bad && threadIdx.x == 0) latch(a.err, PA_ERR_OUT_OF_RANGE);
      for (int i = threadIdx.x; i < Hq * D; i += blockDim.x)
        out[(int64_t)s * Hq * D + i] = Vec<T>::cvt_out(0.f);
    }
  }
  // the attention launch's records and partials are complete past this
  griddep_wait();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    constexpr int kHead = kRecNonEmpty | kRecStart0 | kRecCutEnd;
    int n = 0;
    for (int b = c; b < C; b += 32) {
      const int k = b + lane;
      const int2 r = k < C ? reinterpret_cast<const int2*>(a.ws_rec)[k] : make_int2(0, 0);
      if (b == c) {
        // this CTA's own record: does it hold the start of a cut pair?
        const int f0 = __shfl_sync(0xffffffffu, r.y, 0);
        if ((f0 & kHead) != kHead) break;
        if (lane == 0) {
          pieces[0] = 2 * c + ((f0 & kRecSingle) ? 0 : 1);
          head_pair = r.x;
        }
        n = 1;
      }
      // the CTAs after c that hold a piece, up to the one where the pair ends
      // (the first with a segment that is not a single segment cut at its end)
      const bool has = k > c && (r.y & kRecNonEmpty) != 0;
      const bool ends = has && !((r.y & kRecSingle) && (r.y & kRecCutEnd));
      const unsigned em = __ballot_sync(0xffffffffu, ends);
      const unsigned upto = em ? (em & (0u - em)) * 2u - 1u : 0xffffffffu;
      const unsigned hm = __ballot_sync(0xffffffffu, has) & upto;
      if ((hm >> lane) & 1u) pieces[n + __popc(hm & ((1u << lane) - 1u))] = 2 * k;
      n += __popc(hm);
      if (em) break;
    }
    if (lane == 0) n_pieces = n;
  }
  __syncthreads();
  const int np = n_pieces, pair = head_pair;
  if (np == 0) return;
  const int s = pair / Hkv, kvh = pair - s * Hkv;
  if (pair < 0 || s >= a.num_seqs) return;
  constexpr int PER = (G * D + kMergeThreads - 1) / kMergeThreads;
  float M[PER], Ls[PER], O[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) { M[j] = kNegInfM; Ls[j] = 0.f; O[j] = 0.f; }
  for (int p = 0; p < np; p += 4) {
    float mv[PER][4], lv[PER][4], av[PER][4];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = threadIdx.x + j * kMergeThreads;
      const int g = e / D, d = e - g * D;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        mv[j][u] = kNegInfM; lv[j][u] = 0.f; av[j][u] = 0.f;
        if (p + u < np && e < G * D) {
          const int64_t pk = (int64_t)pieces[p + u] * G + g;
          mv[j][u] = a.ws_ml[2 * pk];
          lv[j][u] = a.ws_ml[2 * pk + 1];
          av[j][u] = a.ws_acc[pk * D + d];
        }
      }
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      float Mn = M[j];
#pragma unroll
      for (int u = 0; u < 4; ++u) Mn = fmaxf(Mn, mv[j][u]);
      if (Mn == kNegInfM) continue;
      const float f = M[j] == kNegInfM ? 0.f : exp2f(M[j] - Mn);
      Ls[j] *= f;
      O[j] *= f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float wt = mv[j][u] == kNegInfM ? 0.f : exp2f(mv[j][u] - Mn);
        Ls[j] += lv[j][u] * wt;
        O[j] += av[j][u] * wt;
      }
      M[j] = Mn;
    }
  }
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = threadIdx.x + j * kMergeThreads;
    if (e >= G * D) break;
    const int g = e / D, d = e - g * D;
    out[((int64_t)s * Hq + (int64_t)kvh * G + g) * D + d] =
        Vec<T>::cvt_out(Ls[j] > 0.f ? O[j] / Ls[j] : 0.f);
  }
}

// ---------------------------------------------------------------- host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
  std::call_once(g_encode_once, []() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// Pool [NB][Hkv][B][D] seen as a 4-D tensor {64, D/64, B, NB*Hkv}: a row of
// D elements split into 128-byte lines. One box is min(B, 64) whole rows of
// one (block, kv head) slice, i.e. one contiguous run of global memory.
bool encode_pool_map(CUtensorMap* map, const void* base, CUtensorMapDataType type,
                     const DecodeArgs& a) {
  const uint64_t D = a.head_size, B = a.block_size;
  const uint64_t planes = (uint64_t)a.num_blocks * a.num_kv_heads;
  if (planes == 0 || planes > 0x7fffffffull) return false;  // signed 32-bit coordinates
  cuuint64_t dims[4] = {64, D / 64, B, planes};
  cuuint64_t strides[3] = {128, D * 2, B * D * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)(D / 64), (cuuint32_t)(B < 64 ? B : 64), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return g_encode(map, type, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp8 pool [NB][Hkv][B][128] of 1-byte codes as a 3-D tensor {128, B, NB*Hkv}
// with the 128-byte swizzle (one row = one line); one box is min(B, 64) whole
// rows of one slice.
bool encode_pool_map_fp8(CUtensorMap* map, const void* base, const DecodeArgs& a) {
  const uint64_t D = a.head_size, B = a.block_size;
  const uint64_t planes = (uint64_t)a.num_blocks * a.num_kv_heads;
  if (planes == 0 || planes > 0x7fffffffull) return false;
  cuuint64_t dims[3] = {D, B, planes};
  cuuint64_t strides[2] = {D, B * D};
  cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)(B < 64 ? B : 64), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int D, int G, bool KV8, bool MULTI, bool SCALED>
constexpr int mma_smem_bytes() {
  constexpr int kSt = ring_stages<KV8, SCALED, MULTI>();
  // 1024-byte alignment, the ring, then barriers, abort flag, tile masks,
  // merge maxima and sums, stage scales (SCALED), the even schedule's start
  // (8-byte aligned: 8 long longs, 2 ints)
  return 1024 + kSt * (2 * kTile * (KV8 ? D : 2 * D) + q_slot_bytes<T, D, G, MULTI>()) +
         2 * kSt * 8 + 4 + 4 * kSt +
         2 * kMmaConsumers * 8 * 4 + 2 * kSt * 8 * 4 + kSt * 4 + 8 + 8 * 8 + 2 * 4 + 16;
}

template <typename T, int D, int G, bool KV8, bool MULTI, bool SCALED>
cudaError_t launch_mma_tdgm(const DecodeArgs& a, float ks, float vs, cudaStream_t st) {
  if (!get_encode()) return cudaErrorNotSupported;
  CUtensorMap tk, tv;
  const bool ok = KV8 ? (encode_pool_map_fp8(&tk, a.kc, a) && encode_pool_map_fp8(&tv, a.vc, a))
                      : (encode_pool_map(&tk, a.kc, MmaOps<T>::kTmaType, a) &&
                         encode_pool_map(&tv, a.vc, MmaOps<T>::kTmaType, a));
  if (!ok) return cudaErrorInvalidValue;
  constexpr int smem = mma_smem_bytes<T, D, G, KV8, MULTI, SCALED>();
  // the CTAs per SM the kernel is built for fit the SM's 228 KB (1 KB of
  // each CTA's shared memory is reserved by the system)
  static_assert(ctas_per_sm<KV8, SCALED, MULTI>() * (smem + 1024) <= 228 * 1024, "shared memory");
  static_assert(2 * kTile * (KV8 ? D : 2 * D) >= kMmaConsumers * 8 * D * 4,
                "an item's merge must fit in one stage");
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, []() {
    attr_err = cudaFuncSetAttribute(decode_mma_kernel<T, D, G, KV8, MULTI, SCALED>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  // one CTA per work item, items_per_cta items each (a CTA walks its items
  // while its producer runs ahead into the next one), or a.even_ctas CTAs
  // sharing the batch's tiles, then the merge of the pairs cut between them
  const int64_t n_items = (int64_t)a.num_splits * a.num_kv_heads * a.num_seqs;
  const bool even = MULTI && a.even_ctas > 0;
  const int per = (MULTI && a.items_per_cta > 1) ? a.items_per_cta : 1;
  const int64_t grid = even ? (int64_t)a.even_ctas : (n_items + per - 1) / per;
  if (grid > 0x7fffffff || grid < 1) return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(decode_mma_kernel<T, D, G, KV8, MULTI, SCALED>, dim3((unsigned)grid),
                             dim3(kMmaThreads), smem, st, a, tk, tv, ks, vs);
  if (e != cudaSuccess) return e;
  if (even) {
    // the merge launch may start while the attention CTAs finish
    // (programmatic dependent launch: its CTAs wait in griddepcontrol.wait
    // before reading what the attention launch wrote)
    return launch_pdl(even_merge_kernel<T, D, G>, dim3((unsigned)grid), dim3(kMergeThreads),
                      (size_t)grid * sizeof(int), st, a);
  }
  return launch_combine(a, st);
}

template <typename T, int D, int G, bool KV8>
cudaError_t launch_mma_tdg(const DecodeArgs& a, float ks, float vs, cudaStream_t st) {
  if constexpr (D == 128) {
    if (a.even_ctas > 0 || a.items_per_cta > 1) {
      if constexpr (KV8) {
        if (a.k_scales != nullptr)
          return launch_mma_tdgm<T, D, G, KV8, true, true>(a, 1.f, 1.f, st);
      }
      return launch_mma_tdgm<T, D, G, KV8, true, false>(a, ks, vs, st);
    }
  }
  if constexpr (KV8) {
    if (a.k_scales != nullptr) return launch_mma_tdgm<T, D, G, KV8, false, true>(a, 1.f, 1.f, st);
  }
  return launch_mma_tdgm<T, D, G, KV8, false, false>(a, ks, vs, st);
}

template <typename T, int D, bool KV8>
cudaError_t launch_mma_td(const DecodeArgs& a, float ks, float vs, cudaStream_t st) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1:
      if constexpr (KV8) return launch_mma_tdg<T, D, 1, KV8>(a, ks, vs, st);
      return cudaErrorInvalidValue;
    case 2: return launch_mma_tdg<T, D, 2, KV8>(a, ks, vs, st);
    case 4: return launch_mma_tdg<T, D, 4, KV8>(a, ks, vs, st);
    case 8: return launch_mma_tdg<T, D, 8, KV8>(a, ks, vs, st);
  }
  return cudaErrorInvalidValue;
}

template <typename T, bool KV8>
cudaError_t launch_mma_t(const DecodeArgs& a, float ks, float vs, cudaStream_t st) {
  if constexpr (!KV8) {
    if (a.head_size == 64) return launch_mma_td<T, 64, false>(a, ks, vs, st);
  }
  if (a.head_size == 128) return launch_mma_td<T, 128, KV8>(a, ks, vs, st);
  return cudaErrorInvalidValue;
}

}  // namespace

bool encode_kv_pool_map(CUtensorMap* map, const void* base, int dtype, int64_t num_blocks,
                        int num_kv_heads, int block_size, int head_size) {
  if (!get_encode()) return false;
  DecodeArgs a{};
  a.num_blocks = num_blocks;
  a.num_kv_heads = num_kv_heads;
  a.block_size = block_size;
  a.head_size = head_size;
  const CUtensorMapDataType t =
      dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return encode_pool_map(map, base, t, a);
}

bool mma_path_applies(const DecodeArgs& a) {
  const int g = a.num_q_heads / a.num_kv_heads;
  return (a.dtype == PA_F16 || a.dtype == PA_BF16) && (g == 2 || g == 4 || g == 8) &&
         a.block_size >= 8 && (a.head_size == 64 || a.head_size == 128);
}

// fp8 pools: the same kernel for every group size with 16-bit queries and
// head size 128, group 1 included (the group is the N = 8 side of the
// products, zero-padded; widening the codes costs the same per byte whatever
// the group, and on the CUDA cores a group of 1 pays a 16-lane reduction per
// token)
bool mma_fp8_path_applies(const DecodeArgs& a) {
  const int g = a.num_q_heads / a.num_kv_heads;
  return (a.dtype == PA_F16 || a.dtype == PA_BF16) && (g == 1 || g == 2 || g == 4 || g == 8) &&
         a.block_size >= 8 && a.head_size == 128;
}

cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t st) {
  if (a.dtype == PA_BF16) return launch_mma_t<__nv_bfloat16, false>(a, 1.f, 1.f, st);
  if (a.dtype == PA_F16) return launch_mma_t<__half, false>(a, 1.f, 1.f, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_mma_fp8(const DecodeArgs& a, float k_scale, float v_scale,
                                  cudaStream_t st) {
  if (a.dtype == PA_BF16) return launch_mma_t<__nv_bfloat16, true>(a, k_scale, v_scale, st);
  if (a.dtype == PA_F16) return launch_mma_t<__half, true>(a, k_scale, v_scale, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
