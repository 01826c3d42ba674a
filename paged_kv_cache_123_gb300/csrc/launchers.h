// Host-side launchers for the kernels, one per translation unit. They assume
// the arguments were validated by the C ABI layer (api.cu) and return a
// cudaError_t from the launch. `sm_count` is the device's multiprocessor
// count; grid-stride kernels cap their grids at 16 CTAs per SM.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

cudaError_t launch_slot_mapping(const int32_t* qsl, int num_reqs,
                                const int64_t* positions, int64_t num_tokens,
                                const int32_t* table, int64_t stride,
                                int block_size, int64_t* slots,
                                cudaStream_t st, int* err);

cudaError_t launch_reshape_and_cache(const void* k, const void* v,
                                     int64_t num_tokens, int num_kv_heads,
                                     int row_bytes, const int64_t* slots,
                                     void* kc, void* vc, int64_t num_blocks,
                                     int block_size, int sm_count, cudaStream_t st,
                                     int* err);

// Up to kCopyMaxLayers layers per launch.
constexpr int kCopyMaxLayers = 64;
cudaError_t launch_copy_blocks(void* const* kcs, void* const* vcs,
                               int num_layers, const int64_t* pairs,
                               int64_t num_pairs, int64_t num_blocks,
                               int64_t block_bytes, cudaStream_t st, int* err);

cudaError_t launch_map_to_kernel_blocks(const int32_t* mtab, int64_t rows, int64_t mstride,
                                        int64_t cols, int r, int32_t* ktab, int64_t kstride,
                                        int sm_count, cudaStream_t st, int* err);

struct DecodeArgs {
  const void* q;
  const void* kc;
  const void* vc;
  const int32_t* tables;
  int64_t table_stride;
  const int32_t* seq_lens;
  int num_seqs, num_q_heads, num_kv_heads, head_size, block_size;
  int64_t num_blocks;
  int dtype;
  float scale;
  int max_seq_len;
  int window;        // sliding window in tokens; 0 = the whole sequence
  int partition;     // tokens per split (multiple of max(64, block_size))
  int num_splits;    // ceil(max_seq_len / partition), >= 1
  // tensor-core decode (head size 128), windowed calls: work items per CTA
  // (<= 1: one each), or the number of CTAs of one wave that share the
  // batch's 64-token tiles evenly (the even schedule; 0 = not used)
  int items_per_cta;
  int even_ctas;
  // fp8 pools whose blocks carry their own scales: [num_blocks][num_kv_heads]
  // fp32 each (nullptr: one scale per pool)
  const float* k_scales;
  const float* v_scales;
  void* out;
  float* ws_acc;     // [S][Hq][num_splits][D]   (num_splits > 1); EVEN: [C][2][G][D]
  float* ws_ml;      // [S][Hq][num_splits][2]   (num_splits > 1); EVEN: [C][2][G][2]
  int* ws_rec;       // EVEN: [C][2] (pair of the CTA's last segment, flags)
  int* err;
};

// Attention dispatch: the tensor-core kernel (decode_mma.cu) for 16-bit
// query-head groups of 2, 4 or 8 with blocks of at least 8 tokens, the
// CUDA-core kernel (decode_simt.cu) otherwise; then the split combine.
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);
// fp8 (E4M3) pools: quantising KV write, and decode attention (q/out dtype
// in a.dtype, caches of 1-byte codes): the tensor-core kernel when
// mma_fp8_path_applies (16-bit queries, head size 128, blocks of at least 8
// tokens, groups of 1, 2, 4 or 8), the CUDA-core kernel of fp8_kv.cu
// otherwise
cudaError_t launch_reshape_and_cache_fp8(const void* k, const void* v, int64_t num_tokens,
                                         int num_kv_heads, int head_size, int dtype,
                                         const int64_t* slots, void* kc, void* vc,
                                         int64_t num_blocks, int block_size, float k_scale,
                                         float v_scale, float* k_scales, float* v_scales,
                                         int sm_count, cudaStream_t st, int* err);
cudaError_t launch_decode_fp8(const DecodeArgs& a, float k_scale, float v_scale,
                              cudaStream_t st);
cudaError_t launch_decode_mma_fp8(const DecodeArgs& a, float k_scale, float v_scale,
                                  cudaStream_t st);
bool mma_path_applies(const DecodeArgs& a);
bool mma_fp8_path_applies(const DecodeArgs& a);
cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t st);
// log-sum-exp combine of the partitions (no-op when num_splits == 1)
cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t st);

// TMA descriptor of a KV pool [num_blocks][num_kv_heads][block_size][head_size]
// (16-bit dtype): boxes of min(block_size, 64) whole rows of one slice.
bool encode_kv_pool_map(CUtensorMap* map, const void* base, int dtype, int64_t num_blocks,
                        int num_kv_heads, int block_size, int head_size);

// Several new tokens per sequence (chunked prefill, speculative tokens):
// causal paged attention, tensor-core kernel (prefill_mma.cu).
struct MultiQueryArgs {
  const void* q;
  const int32_t* qsl;
  int num_seqs;
  const void* kc;
  const void* vc;
  const int32_t* tables;
  int64_t table_stride;
  const int32_t* seq_lens;
  int num_q_heads, num_kv_heads, head_size, block_size;
  int64_t num_blocks;
  int dtype;
  float scale;
  int max_query_len, max_seq_len;
  int64_t num_tokens;  // rows of q / out
  int partition;       // tokens per KV partition
  int num_splits;      // ceil(max_seq_len / partition)
  void* out;
  float* ws_acc;       // [num_tokens][Hq][num_splits][D]   (num_splits > 1)
  float* ws_ml;        // [num_tokens][Hq][num_splits][2]
  int* err;
};
cudaError_t launch_multi_query(const MultiQueryArgs& a, cudaStream_t st);
// The attention launch alone (no partition combine) of the tcgen05 kernel
// for runs of more than 64 (token, head) rows per KV head (prefill_tc.cu).
cudaError_t launch_multi_query_tc(const MultiQueryArgs& a, cudaStream_t st);

}  // namespace pa
