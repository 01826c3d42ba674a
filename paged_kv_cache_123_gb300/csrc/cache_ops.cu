// Slot mapping, KV write (reshape_and_cache) and block copy kernels.
//
// These are the integer / byte-moving steps around paged decode attention:
//   * slot mapping — "PagedAttention 核心创新深度分析" §2.3 (BlockTable and its
//     slot-mapping kernel), single-rank case;
//   * KV write — the new token's K/V rows go to the slot the mapping chose;
//   * block copy — the data movement of block-level copy-on-write
//     ("Visual reading: paged-attention-kv-cache", Figure 8; "Infra:
//     PagedAttention", copy-on-write figure).
// All three are bandwidth-trivial next to attention; they use 16-byte
// vector accesses and never dereference an unchecked index.
#include "common.cuh"
#include "launchers.h"

namespace pa {

// One thread per token. The owning request is found by binary search over
// query_start_loc, so ragged batches (many tokens per request, empty
// requests) need no per-request launch shape.
__global__ void slot_mapping_kernel(const int32_t* __restrict__ qsl, int num_reqs,
                                    const int64_t* __restrict__ positions,
                                    int64_t num_tokens,
                                    const int32_t* __restrict__ table,
                                    int64_t stride, int block_size,
                                    int64_t* __restrict__ slots, int* err) {
  griddep_launch();
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= num_tokens) return;
  griddep_wait();
  // lo = number of entries of qsl[0..num_reqs] that are <= t
  int lo = 0, hi = num_reqs + 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)qsl[mid] <= t) lo = mid + 1; else hi = mid;
  }
  const int r = lo - 1;
  int64_t slot = -1;
  if (r >= 0 && r < num_reqs) {
    const int64_t pos = positions[t];
    const int64_t lb = pos >= 0 ? pos / block_size : -1;
    if (lb < 0 || lb >= stride) {
      latch(err, PA_ERR_OUT_OF_RANGE);
    } else {
      const int64_t pb = table[(int64_t)r * stride + lb];
      if (pb < 0) latch(err, PA_ERR_OUT_OF_RANGE);
      else slot = pb * block_size + (pos - lb * block_size);
    }
  }
  slots[t] = slot;
}

cudaError_t launch_slot_mapping(const int32_t* qsl, int num_reqs,
                                const int64_t* positions, int64_t num_tokens,
                                const int32_t* table, int64_t stride,
                                int block_size, int64_t* slots,
                                cudaStream_t st, int* err) {
  if (num_tokens == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (num_tokens + threads - 1) / threads;
  return launch_pdl(slot_mapping_kernel, dim3((unsigned)blocks), dim3(threads), 0, st, qsl,
                    num_reqs, positions, num_tokens, table, stride, block_size, slots, err);
}

// One thread per 16-byte vector of a (token, kv head) row, K and V together.
__global__ void reshape_and_cache_kernel(const uint4* __restrict__ k,
                                         const uint4* __restrict__ v,
                                         int64_t num_tokens, int num_kv_heads,
                                         int vec_per_row,
                                         const int64_t* __restrict__ slots,
                                         uint4* __restrict__ kc,
                                         uint4* __restrict__ vc,
                                         int64_t num_blocks, int block_size,
                                         int* err) {
  griddep_launch();
  griddep_wait();
  const int64_t n = num_tokens * num_kv_heads * vec_per_row;
  const int64_t limit = num_blocks * block_size;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t c = i % vec_per_row;
    const int64_t th = i / vec_per_row;
    const int64_t h = th % num_kv_heads;
    const int64_t t = th / num_kv_heads;
    const int64_t slot = slots[t];
    if (slot < 0) continue;  // PAD
    if (slot >= limit) {
      if (c == 0 && h == 0) latch(err, PA_ERR_OUT_OF_RANGE);
      continue;
    }
    const int64_t blk = slot / block_size;
    const int64_t row = slot - blk * block_size;
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + row) * vec_per_row + c;
    kc[dst] = k[i];
    vc[dst] = v[i];
  }
}

cudaError_t launch_reshape_and_cache(const void* k, const void* v,
                                     int64_t num_tokens, int num_kv_heads,
                                     int row_bytes, const int64_t* slots,
                                     void* kc, void* vc, int64_t num_blocks,
                                     int block_size, int sm_count, cudaStream_t st,
                                     int* err) {
  if (num_tokens == 0) return cudaSuccess;
  const int vpr = row_bytes / 16;
  const int64_t n = num_tokens * num_kv_heads * vpr;
  const int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  if (blocks > (int64_t)sm_count * 16) blocks = (int64_t)sm_count * 16;
  return launch_pdl(reshape_and_cache_kernel, dim3((unsigned)blocks), dim3(threads), 0, st,
                    (const uint4*)k, (const uint4*)v, num_tokens, num_kv_heads, vpr, slots,
                    (uint4*)kc, (uint4*)vc, num_blocks, block_size, err);
}

struct CopyLayerPtrs {
  char* k[kCopyMaxLayers];
  char* v[kCopyMaxLayers];
};

// grid.z = layer * 2 + {0: K, 1: V}; grid.y strides over pairs; grid.x and
// the threads stride over the 16-byte vectors of one block (W = uint4), or
// over its 4-byte words when the block size is not a multiple of 16 (W =
// uint32_t: the per-block scale arrays of fp8 pools).
template <typename W>
__global__ void copy_blocks_kernel(CopyLayerPtrs p, const int64_t* __restrict__ pairs,
                                   int64_t num_pairs, int64_t num_blocks,
                                   int64_t block_bytes, int* err) {
  const int layer = blockIdx.z >> 1;
  char* base = (blockIdx.z & 1) ? p.v[layer] : p.k[layer];
  const int64_t nvec = block_bytes / (int64_t)sizeof(W);
  for (int64_t pr = blockIdx.y; pr < num_pairs; pr += gridDim.y) {
    const int64_t src = pairs[2 * pr];
    const int64_t dst = pairs[2 * pr + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (threadIdx.x == 0 && blockIdx.x == 0) latch(err, PA_ERR_OUT_OF_RANGE);
      continue;
    }
    const W* s = reinterpret_cast<const W*>(base + src * block_bytes);
    W* d = reinterpret_cast<W*>(base + dst * block_bytes);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec;
         i += (int64_t)gridDim.x * blockDim.x) {
      if constexpr (sizeof(W) == 16)
        d[i] = ld_stream16(s + i);
      else
        d[i] = __ldg(s + i);
    }
  }
}

cudaError_t launch_copy_blocks(void* const* kcs, void* const* vcs,
                               int num_layers, const int64_t* pairs,
                               int64_t num_pairs, int64_t num_blocks,
                               int64_t block_bytes, cudaStream_t st, int* err) {
  if (num_pairs == 0 || num_layers == 0) return cudaSuccess;
  const int threads = 256;
  const bool vec16 = block_bytes % 16 == 0;
  const int64_t nvec = block_bytes / (vec16 ? 16 : 4);
  int64_t gx = (nvec + threads - 1) / threads;
  if (gx > 64) gx = 64;
  const int64_t gy = num_pairs < 65535 ? num_pairs : 65535;
  for (int l0 = 0; l0 < num_layers; l0 += kCopyMaxLayers) {
    const int nl = (num_layers - l0) < kCopyMaxLayers ? (num_layers - l0) : kCopyMaxLayers;
    CopyLayerPtrs p;
    for (int i = 0; i < kCopyMaxLayers; ++i) {
      p.k[i] = i < nl ? (char*)kcs[l0 + i] : nullptr;
      p.v[i] = i < nl ? (char*)vcs[l0 + i] : nullptr;
    }
    dim3 grid((unsigned)gx, (unsigned)gy, (unsigned)(2 * nl));
    if (vec16)
      copy_blocks_kernel<uint4><<<grid, threads, 0, st>>>(p, pairs, num_pairs, num_blocks,
                                                         block_bytes, err);
    else
      copy_blocks_kernel<uint32_t><<<grid, threads, 0, st>>>(p, pairs, num_pairs, num_blocks,
                                                            block_bytes, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pa

namespace pa {

// Hybrid block sizes ("PagedAttention 核心创新深度分析" §3.4,
// map_to_kernel_blocks): the allocator hands out blocks of r kernel blocks;
// its block k owns kernel blocks k*r .. k*r + r - 1. One thread per output
// entry of the expanded table; a negative (unassigned) id stays -1.
__global__ void map_to_kernel_blocks_kernel(const int32_t* __restrict__ mtab, int64_t rows,
                                            int64_t mstride, int64_t cols, int r,
                                            int32_t* __restrict__ ktab, int64_t kstride,
                                            int* err) {
  const int64_t per_row = cols * r;
  const int64_t n = rows * per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / per_row;
    const int64_t j = i - row * per_row;
    const int64_t c = j / r;
    const int64_t k = mtab[row * mstride + c];
    int64_t v = -1;
    if (k >= 0) {
      v = k * r + (j - c * r);
      if (v > 0x7fffffffLL) {
        latch(err, PA_ERR_OUT_OF_RANGE);
        v = -1;
      }
    }
    ktab[row * kstride + j] = (int32_t)v;
  }
}

cudaError_t launch_map_to_kernel_blocks(const int32_t* mtab, int64_t rows, int64_t mstride,
                                        int64_t cols, int r, int32_t* ktab, int64_t kstride,
                                        int sm_count, cudaStream_t st, int* err) {
  const int64_t n = rows * cols * r;
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  if (blocks > (int64_t)sm_count * 16) blocks = (int64_t)sm_count * 16;
  map_to_kernel_blocks_kernel<<<(unsigned)blocks, threads, 0, st>>>(
      mtab, rows, mstride, cols, r, ktab, kstride, err);
  return cudaGetLastError();
}

}  // namespace pa
