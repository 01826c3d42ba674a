// C ABI of libpagedattn.so: argument validation, partition sizing and kernel
// launch. Declarations and their contracts are in include/pagedattn.h.
#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "launchers.h"

// Device-side error word latched by the kernels on bad indices.
static __device__ int g_pa_device_error;

namespace {

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];
int g_dev_status[kMaxDevices];

// Per-device set-up, run once with that device current: the address of the
// error word, its initial clear, and the SM count.
int device_setup(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return PA_ERR_DEVICE;
  std::call_once(g_dev_once[dev], [dev]() {
    int st = PA_OK;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_device_error) != cudaSuccess) st = PA_ERR_DEVICE;
    int zero = 0;
    if (st == PA_OK && cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      st = PA_ERR_DEVICE;
    int sms = 0;
    if (st == PA_OK &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      st = PA_ERR_DEVICE;
    g_err_ptr[dev] = static_cast<int*>(p);
    g_sm_count[dev] = sms > 0 ? sms : 1;
    g_dev_status[dev] = st;
  });
  *dev_out = dev;
  return g_dev_status[dev];
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int elt_bytes(int dtype) {
  switch (dtype) {
    case PA_F32: return 4;
    case PA_F16: return 2;
    case PA_BF16: return 2;
  }
  return 0;
}

int check_launch(cudaError_t e) {
  if (e == cudaSuccess) return PA_OK;
  if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
    return PA_ERR_DEVICE;
  return PA_ERR_CUDA;
}

// Tokens per context partition and the partition count for a batch whose
// longest sequence is max_seq_len. Partitions are whole multiples of
// max(64, block_size) tokens so every partition starts on a block boundary
// and on a 64-token tile. With partition_size == 0 the length is chosen so
// that (sequences x KV heads x partitions) fills two waves of resident CTAs
// even for the longest sequence, then capped: 2048 tokens for the
// tensor-core kernel's shape class (group >= 2, block >= 8; two 100 KB CTAs
// per SM; the fastest of 512..4096 on the GQA batch) and 256 for the
// CUDA-core kernel (many small CTAs per SM, where short partitions even out
// ragged lengths; the fastest of 256..1024 on Llama-7B-shape batches of 32,
// 64 and 128 sequences: 0.99 of the copy bandwidth against 0.96 with 512 at
// 64 sequences, equal at 128).
// uniform = every long sequence covers about max_seq_len tokens (a sliding
// window shorter than the longest sequence): equal work per (sequence, KV
// head), so the partitions are sized for ONE wave of resident CTAs — the
// most splits per pair that still fit — instead of two; a second, partial
// wave would run a few CTAs alone at a fraction of the bandwidth
// (longctx-shaped window of 4096: 0.68 -> 0.80 of the copy bandwidth; a
// 333-token window over the Llama-7B batch: 0.85 -> 0.92).
// mma_fp8 = the call runs the tensor-core kernel over fp8 pools, which takes
// the tensor-core class for every group size (group 1 included: one
// 2,048-token partition per Llama-7B sequence ran at 0.81 of the copy
// bandwidth, 512-token ones at 0.69). That kernel runs three CTAs per SM, so
// a windowed (uniform) call sizes its one wave for three CTAs per SM; more,
// shorter partitions were slower (each item pays its start and its merge:
// a 4096-token window over the long-context batch ran at 0.53 of the copy
// bandwidth with 3 splits, 0.49 with 2 and 0.50 with 7; a 1000-token window
// over the GQA batch at 0.56 unsplit, 0.46 with 2).
void partitioning(int num_seqs, int num_q_heads, int num_kv_heads, int block_size,
                  int max_seq_len, int partition_size, int sm_count, bool uniform,
                  bool mma_fp8, int* splits, int* tokens) {
  const int64_t tile = block_size > 64 ? block_size : 64;
  const int64_t len = max_seq_len > 0 ? max_seq_len : 1;
  auto round_up = [tile](int64_t x) { return (x + tile - 1) / tile * tile; };
  int64_t P;
  if (partition_size > 0) {
    P = round_up(partition_size);
  } else {
    const int g = num_q_heads / num_kv_heads;
    const bool tc = (g >= 2 && block_size >= 8) || mma_fp8;
    const int64_t per_sm = tc ? 2 : 8;
    const int64_t cap = round_up(tc ? 2048 : 256);
    const int64_t pairs = num_seqs > 0 ? (int64_t)num_seqs * num_kv_heads : 1;
    const int64_t floor_p = round_up(256);
    if (uniform) {
      // splits per pair in one wave (the fp8 kernel runs three CTAs per SM)
      int64_t k = (int64_t)sm_count * (mma_fp8 ? 3 : per_sm) / pairs;
      if (k < 1) k = 1;
      P = round_up((len + k - 1) / k);
      if (P < floor_p) P = floor_p;
    } else {
      const int64_t target = 2 * (int64_t)sm_count * per_sm;
      P = round_up((len * pairs + target - 1) / target);
      if (P < floor_p) P = floor_p;
      if (P > cap) P = cap;
    }
  }
  if (P > len) P = round_up(len);
  if (P > (int64_t)1 << 30) P = (int64_t)1 << 30;
  *tokens = (int)P;
  *splits = (int)((len + P - 1) / P);
}

int64_t workspace_for(int num_seqs, int num_q_heads, int head_size, int splits) {
  if (splits <= 1) return 0;
  const int64_t n = (int64_t)num_seqs * num_q_heads * splits;
  const int64_t acc = n * head_size * 4;
  const int64_t ml = n * 2 * 4;
  return ((acc + 255) / 256) * 256 + ml;
}

// Longest token range one sequence's partitions cover: with a sliding
// window the range starts at the window's first token rounded down to a
// 64-token tile (the kernels' window_base), so it spans at most
// window + 63 tokens.
int covered_len(int max_seq_len, int window) {
  if (window <= 0 || window >= max_seq_len) return max_seq_len;
  return std::min<int64_t>(max_seq_len, (int64_t)window + 63);
}

// A window that cuts the longest sequence: every sequence at least that long
// covers window .. window + 63 tokens.
bool windowed(int max_seq_len, int window) { return window > 0 && window < max_seq_len; }

// Windowed tensor-core decode calls (head size 128) with automatic
// partitioning run one wave of resident CTAs (2 per SM for 16-bit pools, 3
// for fp8 pools; the kernel's CTAs that walk several items run three per
// SM with per-block scales too).
// A window cuts every long sequence to about the same work, and the fixed
// partitions give items of equal length: when there are more items than
// slots, each CTA walks several (items_per_cta, strided). Whole items rarely
// divide evenly over the slots: with per = ceil(items / slots) items per
// CTA, the busiest CTA does imbalance = per * slots / items times the mean
// work. Above kEvenImbalance the even schedule takes over: the batch's
// 64-token tiles (all (sequence, KV head) pairs in order) are cut into C
// equal consecutive runs, one per CTA, and a merge launch combines the pairs
// cut between CTAs. Measured on GB300: the GQA-72B batch with a 1000-token
// window over fp8 pools (1,024 items for 456 slots, imbalance 1.34) went
// from 0.57 to 0.63 of the copy bandwidth; at imbalance 1.19 or below (the
// same window over 16-bit pools, the long-context batch with a 4096-token
// window, the Llama-7B batch with a 333-token window over fp8 pools) the
// merge launch cost as much as the balance gained or more.
// The start of a CTA's share is found by a pass over the sequence lengths
// in every CTA, so the even schedule is kept to batches of at most
// kEvenMaxSeqs sequences.
constexpr int kEvenMaxSeqs = 8192;
constexpr double kEvenImbalance = 1.25;
bool even_applies(int num_seqs, int head_size, int max_seq_len, int window, int partition_size,
                  bool tc_path) {
  return tc_path && head_size == 128 && partition_size == 0 && windowed(max_seq_len, window) &&
         num_seqs <= kEvenMaxSeqs;
}
// For a call where even_applies: the items per CTA of the strided walk
// (items_per_cta) or the CTA count of the even schedule (even_ctas > 0).
void wave_plan(int num_seqs, int num_kv_heads, int splits, int max_seq_len, int window,
               int sm_count, int ctas_per_sm, int* items_per_cta, int64_t* even_ctas) {
  const int64_t items = (int64_t)splits * num_kv_heads * num_seqs;
  const int64_t slots = (int64_t)sm_count * ctas_per_sm;
  const int64_t per = std::max<int64_t>(1, (items + slots - 1) / slots);
  *items_per_cta = (int)std::min<int64_t>(1 << 20, per);
  *even_ctas = 0;
  if (items > 0 && (double)(per * slots) > kEvenImbalance * (double)items) {
    const int64_t tiles_per_pair = ((int64_t)covered_len(max_seq_len, window) + 63) / 64;
    const int64_t upper = (int64_t)num_seqs * num_kv_heads * tiles_per_pair;
    *even_ctas = std::max<int64_t>(1, std::min(slots, upper));
    *items_per_cta = 1;
  }
}
// partial outputs [C][2][G][D], maxima and sums [C][2][G][2], records [C][2]
int64_t even_workspace(int64_t ctas, int group, int head_size) {
  const int64_t acc = ctas * 2 * group * head_size * 4;
  const int64_t ml = ctas * 2 * group * 2 * 4;
  return ((acc + 255) / 256) * 256 + ((ml + 255) / 256) * 256 + ctas * 2 * 4;
}

int decode_partitioning(int num_seqs, int num_q_heads, int num_kv_heads, int block_size,
                        int max_seq_len, int window, int partition_size, bool mma_fp8,
                        int* splits, int* tokens);

// Validation, partitioning and launch shared by the decode entry points
// (16-bit/fp32 pools or E4M3 pools, with or without a window).
int run_decode(const void* q, const void* key_cache, const void* value_cache,
               const int32_t* block_tables, int64_t block_tables_stride,
               const int32_t* seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
               int head_size, int block_size, int64_t num_blocks, int dtype, float scale,
               bool fp8, float k_scale, float v_scale, const float* k_scales,
               const float* v_scales, int window, int max_seq_len, int partition_size,
               void* out, void* workspace, int64_t workspace_bytes, void* stream);

int check_decode_shape(int num_seqs, int num_q_heads, int num_kv_heads, int head_size,
                       int block_size, int max_seq_len) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_seq_len < 0)
    return PA_ERR_SHAPE;
  if (head_size != 64 && head_size != 128) return PA_ERR_SHAPE;
  if (!pow2(block_size) || block_size > 256) return PA_ERR_SHAPE;
  if (num_q_heads % num_kv_heads != 0) return PA_ERR_SHAPE;
  const int g = num_q_heads / num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return PA_ERR_SHAPE;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_SHAPE;
  return PA_OK;
}

// Partitioning of a decode call over max_seq_len (and a window, 0 = none),
// with the device's SM count.
int decode_partitioning(int num_seqs, int num_q_heads, int num_kv_heads, int block_size,
                        int max_seq_len, int window, int partition_size, bool mma_fp8,
                        int* splits, int* tokens) {
  if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 ||
      num_q_heads % num_kv_heads != 0 || !pow2(block_size) || block_size > 256 ||
      max_seq_len < 0 || partition_size < 0 || window < 0)
    return PA_ERR_SHAPE;
  int dev;
  int st = device_setup(&dev);
  if (st != PA_OK) return st;
  int sp, tk;
  partitioning(num_seqs, num_q_heads, num_kv_heads, block_size,
               covered_len(max_seq_len, window), partition_size, g_sm_count[dev],
               windowed(max_seq_len, window), mma_fp8, &sp, &tk);
  if (splits) *splits = sp;
  if (tokens) *tokens = tk;
  return PA_OK;
}

}  // namespace

extern "C" {

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_NULL: return "a required pointer is NULL";
    case PA_ERR_SHAPE: return "unsupported or inconsistent size";
    case PA_ERR_DTYPE: return "unknown dtype code";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_OUT_OF_RANGE: return "an index is outside its array";
    case PA_ERR_CUDA: return "CUDA runtime call or launch failed";
    case PA_ERR_ALIAS: return "copy pairs overlap";
    case PA_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case PA_ERR_DEVICE: return "no usable sm_103 device or kernel image";
    case PA_ERR_TIMEOUT: return "a kernel gave up waiting on an asynchronous copy";
  }
  return "unknown status";
}

int pa_abi_version(void) { return 2; }

int pa_compute_slot_mapping(const int32_t* query_start_loc, int num_reqs,
                            const int64_t* positions, int64_t num_tokens,
                            const int32_t* block_table, int64_t block_table_stride,
                            int block_size, int64_t* slot_mapping, void* stream) {
  if (num_reqs < 0 || num_tokens < 0 || block_size <= 0 || block_table_stride < 0)
    return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!query_start_loc || !positions || !slot_mapping) return PA_ERR_NULL;
  if (num_reqs > 0 && !block_table) return PA_ERR_NULL;
  int dev;
  int st = device_setup(&dev);
  if (st != PA_OK) return st;
  return check_launch(pa::launch_slot_mapping(
      query_start_loc, num_reqs, positions, num_tokens, block_table,
      block_table_stride, block_size, slot_mapping, (cudaStream_t)stream, g_err_ptr[dev]));
}

int pa_reshape_and_cache(const void* k, const void* v, int64_t num_tokens,
                         int num_kv_heads, int head_size, int dtype,
                         const int64_t* slot_mapping, void* key_cache,
                         void* value_cache, int64_t num_blocks, int block_size,
                         void* stream) {
  const int eb = elt_bytes(dtype);
  if (eb == 0) return PA_ERR_DTYPE;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 ||
      num_blocks < 0)
    return PA_ERR_SHAPE;
  if (((int64_t)head_size * eb) % 16 != 0) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !key_cache || !value_cache) return PA_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(key_cache) || !aligned16(value_cache))
    return PA_ERR_ALIGN;
  int dev;
  int st = device_setup(&dev);
  if (st != PA_OK) return st;
  return check_launch(pa::launch_reshape_and_cache(
      k, v, num_tokens, num_kv_heads, head_size * eb, slot_mapping, key_cache,
      value_cache, num_blocks, block_size, g_sm_count[dev], (cudaStream_t)stream,
      g_err_ptr[dev]));
}

int pa_decode_partitioning(int num_seqs, int num_q_heads, int num_kv_heads, int block_size,
                           int max_seq_len, int partition_size,
                           int* num_splits_out, int* partition_tokens_out) {
  return decode_partitioning(num_seqs, num_q_heads, num_kv_heads, block_size, max_seq_len, 0,
                             partition_size, false, num_splits_out, partition_tokens_out);
}

int pa_decode_window_partitioning(int num_seqs, int num_q_heads, int num_kv_heads,
                                  int block_size, int max_seq_len, int window,
                                  int partition_size, int* num_splits_out,
                                  int* partition_tokens_out) {
  if (window < 0) return PA_ERR_SHAPE;
  return decode_partitioning(num_seqs, num_q_heads, num_kv_heads, block_size, max_seq_len,
                             window, partition_size, false, num_splits_out, partition_tokens_out);
}

int pa_decode_fp8_partitioning(int num_seqs, int num_q_heads, int num_kv_heads, int head_size,
                               int block_size, int dtype, int max_seq_len, int window,
                               int partition_size, int* num_splits_out,
                               int* partition_tokens_out) {
  if (elt_bytes(dtype) == 0) return PA_ERR_DTYPE;
  if (window < 0 || num_kv_heads <= 0) return PA_ERR_SHAPE;
  pa::DecodeArgs a{};
  a.num_q_heads = num_q_heads; a.num_kv_heads = num_kv_heads;
  a.head_size = head_size; a.block_size = block_size; a.dtype = dtype;
  return decode_partitioning(num_seqs, num_q_heads, num_kv_heads, block_size, max_seq_len,
                             window, partition_size, pa::mma_fp8_path_applies(a),
                             num_splits_out, partition_tokens_out);
}

int pa_decode_even_ctas(int num_seqs, int num_q_heads, int num_kv_heads, int head_size,
                        int block_size, int dtype, int kv_format, int max_seq_len, int window,
                        int partition_size) {
  if (elt_bytes(dtype) == 0) return PA_ERR_DTYPE;
  if (kv_format < 0 || kv_format > 2 || window < 0 || partition_size < 0) return PA_ERR_SHAPE;
  int st = check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                              max_seq_len);
  if (st != PA_OK) return st;
  pa::DecodeArgs a{};
  a.num_q_heads = num_q_heads; a.num_kv_heads = num_kv_heads;
  a.head_size = head_size; a.block_size = block_size; a.dtype = dtype;
  const bool tc = kv_format == 0 ? pa::mma_path_applies(a) : pa::mma_fp8_path_applies(a);
  if (num_seqs == 0 ||
      !even_applies(num_seqs, head_size, max_seq_len, window, partition_size, tc))
    return 0;
  int splits, tokens;
  st = decode_partitioning(num_seqs, num_q_heads, num_kv_heads, block_size, max_seq_len, window,
                           partition_size, kv_format != 0, &splits, &tokens);
  if (st != PA_OK) return st;
  int dev;
  st = device_setup(&dev);
  if (st != PA_OK) return st;
  int per;
  int64_t C;
  wave_plan(num_seqs, num_kv_heads, splits, max_seq_len, window, g_sm_count[dev],
            kv_format == 0 ? 2 : 3, &per, &C);
  return (int)C;
}

int64_t pa_decode_fp8_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                      int head_size, int block_size, int dtype,
                                      int max_seq_len, int window, int partition_size) {
  if (elt_bytes(dtype) == 0) return PA_ERR_DTYPE;
  if (window < 0 || partition_size < 0) return PA_ERR_SHAPE;
  int st = check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_size,
                              block_size, max_seq_len);
  if (st != PA_OK) return st;
  pa::DecodeArgs a{};
  a.num_q_heads = num_q_heads; a.num_kv_heads = num_kv_heads;
  a.head_size = head_size; a.block_size = block_size; a.dtype = dtype;
  int splits, tokens;
  const bool tc8 = pa::mma_fp8_path_applies(a);
  st = decode_partitioning(num_seqs, num_q_heads, num_kv_heads, block_size, max_seq_len, window,
                           partition_size, tc8, &splits, &tokens);
  if (st != PA_OK) return st;
  int64_t ws = workspace_for(num_seqs, num_q_heads, head_size, splits);
  if (even_applies(num_seqs, head_size, max_seq_len, window, partition_size, tc8)) {
    // the even schedule, if the call takes it
    int dev;
    st = device_setup(&dev);
    if (st != PA_OK) return st;
    int per;
    int64_t C;
    wave_plan(num_seqs, num_kv_heads, splits, max_seq_len, window, g_sm_count[dev], 3, &per,
              &C);
    if (C > 0) ws = std::max(ws, even_workspace(C, num_q_heads / num_kv_heads, head_size));
  }
  return ws;
}

int64_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                  int head_size, int block_size, int max_seq_len,
                                  int partition_size) {
  int st = check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_size,
                              block_size, max_seq_len);
  if (st != PA_OK) return st;
  if (partition_size < 0) return PA_ERR_SHAPE;
  int splits, tokens;
  st = decode_partitioning(num_seqs, num_q_heads, num_kv_heads, block_size, max_seq_len, 0,
                           partition_size, false, &splits, &tokens);
  if (st != PA_OK) return st;
  return workspace_for(num_seqs, num_q_heads, head_size, splits);
}

int pa_decode_attention(const void* q, const void* key_cache, const void* value_cache,
                        const int32_t* block_tables, int64_t block_tables_stride,
                        const int32_t* seq_lens, int num_seqs, int num_q_heads,
                        int num_kv_heads, int head_size, int block_size,
                        int64_t num_blocks, int dtype, float scale, int max_seq_len,
                        int partition_size, void* out, void* workspace,
                        int64_t workspace_bytes, void* stream) {
  return run_decode(q, key_cache, value_cache, block_tables, block_tables_stride, seq_lens,
                    num_seqs, num_q_heads, num_kv_heads, head_size, block_size, num_blocks,
                    dtype, scale, false, 1.f, 1.f, nullptr, nullptr, 0, max_seq_len, partition_size, out,
                    workspace, workspace_bytes, stream);
}

int64_t pa_decode_window_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                         int head_size, int block_size, int max_seq_len,
                                         int window, int partition_size) {
  if (window < 0) return PA_ERR_SHAPE;
  int st = check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_size,
                              block_size, max_seq_len);
  if (st != PA_OK) return st;
  if (partition_size < 0) return PA_ERR_SHAPE;
  int splits, tokens;
  st = decode_partitioning(num_seqs, num_q_heads, num_kv_heads, block_size, max_seq_len, window,
                           partition_size, false, &splits, &tokens);
  if (st != PA_OK) return st;
  const int64_t fixed = workspace_for(num_seqs, num_q_heads, head_size, splits);
  // 16-bit queries of the tensor-core shape class take the even schedule,
  // fp32 queries the partitions: enough for either
  pa::DecodeArgs a{};
  a.num_q_heads = num_q_heads; a.num_kv_heads = num_kv_heads;
  a.head_size = head_size; a.block_size = block_size; a.dtype = PA_BF16;
  if (even_applies(num_seqs, head_size, max_seq_len, window, partition_size,
                   pa::mma_path_applies(a))) {
    int dev;
    st = device_setup(&dev);
    if (st != PA_OK) return st;
    int per;
    int64_t C;
    wave_plan(num_seqs, num_kv_heads, splits, max_seq_len, window, g_sm_count[dev], 2, &per,
              &C);
    if (C > 0) return std::max(fixed, even_workspace(C, num_q_heads / num_kv_heads, head_size));
  }
  return fixed;
}

int pa_decode_attention_window(const void* q, const void* key_cache, const void* value_cache,
                               const int32_t* block_tables, int64_t block_tables_stride,
                               const int32_t* seq_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_size, int block_size,
                               int64_t num_blocks, int dtype, float scale, int window,
                               int max_seq_len, int partition_size, void* out,
                               void* workspace, int64_t workspace_bytes, void* stream) {
  if (window < 0) return PA_ERR_SHAPE;
  return run_decode(q, key_cache, value_cache, block_tables, block_tables_stride, seq_lens,
                    num_seqs, num_q_heads, num_kv_heads, head_size, block_size, num_blocks,
                    dtype, scale, false, 1.f, 1.f, nullptr, nullptr, window, max_seq_len, partition_size, out,
                    workspace, workspace_bytes, stream);
}

// Context partitions of the multi-query kernels. Only short query runs (at
// most 64 (token, head) rows per KV head, e.g. speculative tokens) are
// split: longer runs already give many row tiles. Runs of 17..64 rows go to
// the tcgen05 kernel, one CTA per SM whose start-up is not hidden by a
// neighbour: partitions only as short as needed for one CTA per SM (4 and 8
// speculative tokens over the GQA-72B batch: 0.82 / 0.74 of the copy
// bandwidth with 2,048-token partitions, 0.94 / 0.92 unsplit). Runs of at
// most 16 rows (the mma.sync column kernel, two CTAs per SM) are split only
// as far as one wave of those needs (2 speculative tokens: 0.87 with
// 2,048-token partitions, 0.90 unsplit).
static void mq_partitioning(int num_seqs, int num_q_heads, int num_kv_heads, int block_size,
                     int max_query_len, int max_seq_len, int partition_size, int sm_count,
                     int* splits, int* tokens) {
  const int g = num_q_heads / num_kv_heads;
  const int64_t tile = block_size > 64 ? block_size : 64;
  const int64_t len = max_seq_len > 0 ? max_seq_len : 1;
  auto round_up = [tile](int64_t x) { return (x + tile - 1) / tile * tile; };
  int64_t P;
  if (partition_size > 0) {
    P = round_up(partition_size);
  } else if ((int64_t)max_query_len * g > 64) {
    P = round_up(len);
  } else {
    // one wave: one tcgen05 CTA per SM, or two column-kernel CTAs per SM
    const int64_t ctas = num_seqs > 0 ? (int64_t)num_seqs * num_kv_heads : 1;
    const int64_t slots = (int64_t)sm_count * ((int64_t)max_query_len * g > 16 ? 1 : 2);
    P = round_up((len * ctas + slots - 1) / slots);
    if (P < round_up(256)) P = round_up(256);
  }
  if (P > len) P = round_up(len);
  *tokens = (int)P;
  *splits = (int)((len + P - 1) / P);
}

static int check_mq_shape(int num_seqs, int num_q_heads, int num_kv_heads, int head_size,
                   int block_size, int max_query_len, int max_seq_len) {
  int st = check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                              max_seq_len);
  if (st != PA_OK) return st;
  if (block_size < 8 || max_query_len < 0) return PA_ERR_SHAPE;
  if ((int64_t)max_query_len * (num_q_heads / num_kv_heads) > 0x7fffffffll) return PA_ERR_SHAPE;
  return PA_OK;
}

int64_t pa_multi_query_workspace_bytes(int64_t num_tokens, int num_seqs, int num_q_heads,
                                       int num_kv_heads, int head_size, int block_size,
                                       int max_query_len, int max_seq_len, int partition_size) {
  int st = check_mq_shape(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                          max_query_len, max_seq_len);
  if (st != PA_OK) return st;
  if (num_tokens < 0 || partition_size < 0) return PA_ERR_SHAPE;
  int dev;
  st = device_setup(&dev);
  if (st != PA_OK) return st;
  int splits, tokens;
  mq_partitioning(num_seqs, num_q_heads, num_kv_heads, block_size, max_query_len, max_seq_len,
                  partition_size, g_sm_count[dev], &splits, &tokens);
  if (splits <= 1) return 0;
  const int64_t n = num_tokens * num_q_heads * splits;
  return ((n * head_size * 4 + 255) / 256) * 256 + n * 2 * 4;
}

int pa_multi_query_attention(const void* q, const int32_t* query_start_loc, int num_seqs,
                             int64_t num_tokens, const void* key_cache, const void* value_cache,
                             const int32_t* block_tables, int64_t block_tables_stride,
                             const int32_t* seq_lens, int num_q_heads, int num_kv_heads,
                             int head_size, int block_size, int64_t num_blocks, int dtype,
                             float scale, int max_query_len, int max_seq_len,
                             int partition_size, void* out, void* workspace,
                             int64_t workspace_bytes, void* stream) {
  if (dtype != PA_F16 && dtype != PA_BF16) return elt_bytes(dtype) ? PA_ERR_SHAPE : PA_ERR_DTYPE;
  int st = check_mq_shape(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                          max_query_len, max_seq_len);
  if (st != PA_OK) return st;
  if (num_blocks < 0 || block_tables_stride < 0 || num_tokens < 0 || partition_size < 0)
    return PA_ERR_SHAPE;
  if ((int64_t)max_seq_len > block_tables_stride * block_size) return PA_ERR_OUT_OF_RANGE;
  if (num_seqs == 0 || max_query_len == 0 || num_tokens == 0) return PA_OK;
  if (!q || !query_start_loc || !key_cache || !value_cache || !block_tables || !seq_lens || !out)
    return PA_ERR_NULL;
  if (!aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache) || !aligned16(out))
    return PA_ERR_ALIGN;
  int dev;
  st = device_setup(&dev);
  if (st != PA_OK) return st;
  pa::MultiQueryArgs a;
  a.q = q; a.qsl = query_start_loc; a.num_seqs = num_seqs; a.num_tokens = num_tokens;
  a.kc = key_cache; a.vc = value_cache; a.tables = block_tables;
  a.table_stride = block_tables_stride; a.seq_lens = seq_lens;
  a.num_q_heads = num_q_heads; a.num_kv_heads = num_kv_heads; a.head_size = head_size;
  a.block_size = block_size; a.num_blocks = num_blocks; a.dtype = dtype; a.scale = scale;
  a.max_query_len = max_query_len; a.max_seq_len = max_seq_len; a.out = out;
  mq_partitioning(num_seqs, num_q_heads, num_kv_heads, block_size, max_query_len, max_seq_len,
                  partition_size, g_sm_count[dev], &a.num_splits, &a.partition);
  a.ws_acc = nullptr; a.ws_ml = nullptr;
  if (a.num_splits > 1) {
    const int64_t n = num_tokens * num_q_heads * a.num_splits;
    const int64_t acc = ((n * head_size * 4 + 255) / 256) * 256;
    if (!workspace || workspace_bytes < acc + n * 8) return PA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PA_ERR_ALIGN;
    a.ws_acc = static_cast<float*>(workspace);
    a.ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc);
  }
  a.err = g_err_ptr[dev];
  return check_launch(pa::launch_multi_query(a, (cudaStream_t)stream));
}

int pa_reshape_and_cache_fp8(const void* k, const void* v, int64_t num_tokens, int num_kv_heads,
                             int head_size, int dtype, const int64_t* slot_mapping,
                             void* key_cache, void* value_cache, int64_t num_blocks,
                             int block_size, float k_scale, float v_scale, void* stream) {
  if (elt_bytes(dtype) == 0) return PA_ERR_DTYPE;
  if (num_tokens < 0 || num_kv_heads <= 0 || block_size <= 0 || num_blocks < 0 ||
      head_size <= 0 || head_size % 16 != 0)
    return PA_ERR_SHAPE;
  if (!(k_scale > 0.f) || !(v_scale > 0.f)) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !key_cache || !value_cache) return PA_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(key_cache) || !aligned16(value_cache))
    return PA_ERR_ALIGN;
  int dev;
  int st = device_setup(&dev);
  if (st != PA_OK) return st;
  return check_launch(pa::launch_reshape_and_cache_fp8(
      k, v, num_tokens, num_kv_heads, head_size, dtype, slot_mapping, key_cache, value_cache,
      num_blocks, block_size, k_scale, v_scale, nullptr, nullptr, g_sm_count[dev],
      (cudaStream_t)stream, g_err_ptr[dev]));
}

int pa_reshape_and_cache_fp8_scaled(const void* k, const void* v, int64_t num_tokens,
                                    int num_kv_heads, int head_size, int dtype,
                                    const int64_t* slot_mapping, void* key_cache,
                                    void* value_cache, float* k_scales, float* v_scales,
                                    int64_t num_blocks, int block_size, void* stream) {
  if (elt_bytes(dtype) == 0) return PA_ERR_DTYPE;
  if (num_tokens < 0 || num_kv_heads <= 0 || block_size <= 0 || num_blocks < 0 ||
      head_size <= 0 || head_size % 16 != 0)
    return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !key_cache || !value_cache || !k_scales || !v_scales)
    return PA_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(key_cache) || !aligned16(value_cache) ||
      !aligned16(k_scales) || !aligned16(v_scales))
    return PA_ERR_ALIGN;
  int dev;
  int st = device_setup(&dev);
  if (st != PA_OK) return st;
  return check_launch(pa::launch_reshape_and_cache_fp8(
      k, v, num_tokens, num_kv_heads, head_size, dtype, slot_mapping, key_cache, value_cache,
      num_blocks, block_size, 1.f, 1.f, k_scales, v_scales, g_sm_count[dev],
      (cudaStream_t)stream, g_err_ptr[dev]));
}

int pa_decode_attention_fp8(const void* q, const void* key_cache, const void* value_cache,
                            const int32_t* block_tables, int64_t block_tables_stride,
                            const int32_t* seq_lens, int num_seqs, int num_q_heads,
                            int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
                            int dtype, float scale, float k_scale, float v_scale,
                            int max_seq_len, int partition_size, void* out, void* workspace,
                            int64_t workspace_bytes, void* stream) {
  return run_decode(q, key_cache, value_cache, block_tables, block_tables_stride, seq_lens,
                    num_seqs, num_q_heads, num_kv_heads, head_size, block_size, num_blocks,
                    dtype, scale, true, k_scale, v_scale, nullptr, nullptr, 0, max_seq_len, partition_size, out,
                    workspace, workspace_bytes, stream);
}

int pa_decode_attention_fp8_scaled(const void* q, const void* key_cache,
                                   const void* value_cache, const float* k_scales,
                                   const float* v_scales, const int32_t* block_tables,
                                   int64_t block_tables_stride, const int32_t* seq_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads,
                                   int head_size, int block_size, int64_t num_blocks, int dtype,
                                   float scale, int window, int max_seq_len, int partition_size,
                                   void* out, void* workspace, int64_t workspace_bytes,
                                   void* stream) {
  if (window < 0) return PA_ERR_SHAPE;
  if (num_seqs > 0 && (!k_scales || !v_scales)) return PA_ERR_NULL;
  return run_decode(q, key_cache, value_cache, block_tables, block_tables_stride, seq_lens,
                    num_seqs, num_q_heads, num_kv_heads, head_size, block_size, num_blocks,
                    dtype, scale, true, 1.f, 1.f, k_scales, v_scales, window, max_seq_len,
                    partition_size, out, workspace, workspace_bytes, stream);
}

int pa_decode_attention_fp8_window(const void* q, const void* key_cache,
                                   const void* value_cache, const int32_t* block_tables,
                                   int64_t block_tables_stride, const int32_t* seq_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads,
                                   int head_size, int block_size, int64_t num_blocks, int dtype,
                                   float scale, float k_scale, float v_scale, int window,
                                   int max_seq_len, int partition_size, void* out,
                                   void* workspace, int64_t workspace_bytes, void* stream) {
  if (window < 0) return PA_ERR_SHAPE;
  return run_decode(q, key_cache, value_cache, block_tables, block_tables_stride, seq_lens,
                    num_seqs, num_q_heads, num_kv_heads, head_size, block_size, num_blocks,
                    dtype, scale, true, k_scale, v_scale, nullptr, nullptr, window, max_seq_len, partition_size,
                    out, workspace, workspace_bytes, stream);
}

int pa_copy_blocks(void* const* key_caches, void* const* value_caches, int num_layers,
                   const int64_t* src_dst_pairs, const int64_t* src_dst_pairs_host,
                   int64_t num_pairs, int64_t num_blocks, int64_t block_bytes,
                   void* stream) {
  if (num_layers < 0 || num_pairs < 0 || num_blocks < 0) return PA_ERR_SHAPE;
  if (block_bytes <= 0 || block_bytes % 4 != 0) return PA_ERR_SHAPE;
  if (num_pairs == 0 || num_layers == 0) return PA_OK;
  if (!key_caches || !value_caches || !src_dst_pairs) return PA_ERR_NULL;
  for (int l = 0; l < num_layers; ++l) {
    if (!key_caches[l] || !value_caches[l]) return PA_ERR_NULL;
    if (!aligned16(key_caches[l]) || !aligned16(value_caches[l])) return PA_ERR_ALIGN;
  }
  if (src_dst_pairs_host) {
    // ranges, then aliasing: sort-free O(P log P) via a sorted copy
    std::vector<int64_t> d, s;
    d.reserve(num_pairs); s.reserve(num_pairs);
    for (int64_t i = 0; i < num_pairs; ++i) {
      const int64_t a = src_dst_pairs_host[2 * i], b = src_dst_pairs_host[2 * i + 1];
      if (a < 0 || a >= num_blocks || b < 0 || b >= num_blocks) return PA_ERR_OUT_OF_RANGE;
      s.push_back(a); d.push_back(b);
    }
    std::sort(d.begin(), d.end());
    std::sort(s.begin(), s.end());
    for (int64_t i = 1; i < num_pairs; ++i)
      if (d[i] == d[i - 1]) return PA_ERR_ALIAS;
    for (int64_t x : d)
      if (std::binary_search(s.begin(), s.end(), x)) return PA_ERR_ALIAS;
  }
  int dev;
  int st = device_setup(&dev);
  if (st != PA_OK) return st;
  return check_launch(pa::launch_copy_blocks(key_caches, value_caches, num_layers,
                                             src_dst_pairs, num_pairs, num_blocks,
                                             block_bytes, (cudaStream_t)stream,
                                             g_err_ptr[dev]));
}

int pa_map_to_kernel_blocks(const int32_t* manager_table, int64_t num_rows,
                            int64_t manager_stride, int64_t num_cols, int blocks_per_kv_block,
                            int32_t* kernel_table, int64_t kernel_stride, void* stream) {
  if (num_rows < 0 || num_cols < 0 || blocks_per_kv_block < 1 || manager_stride < num_cols ||
      kernel_stride < num_cols * blocks_per_kv_block)
    return PA_ERR_SHAPE;
  if (num_rows == 0 || num_cols == 0) return PA_OK;
  if (!manager_table || !kernel_table) return PA_ERR_NULL;
  int dev;
  int st = device_setup(&dev);
  if (st != PA_OK) return st;
  return check_launch(pa::launch_map_to_kernel_blocks(
      manager_table, num_rows, manager_stride, num_cols, blocks_per_kv_block, kernel_table,
      kernel_stride, g_sm_count[dev], (cudaStream_t)stream, g_err_ptr[dev]));
}

int pa_get_device_error(int* code_out, void* stream) {
  if (!code_out) return PA_ERR_NULL;
  int dev;
  int st = device_setup(&dev);
  if (st != PA_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  int v = 0, zero = 0;
  if (cudaMemcpyAsync(&v, g_err_ptr[dev], sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaMemcpyAsync(g_err_ptr[dev], &zero, sizeof(int), cudaMemcpyHostToDevice, s) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  *code_out = v;
  return PA_OK;
}

}  // extern "C"

namespace {

int run_decode(const void* q, const void* key_cache, const void* value_cache,
               const int32_t* block_tables, int64_t block_tables_stride,
               const int32_t* seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
               int head_size, int block_size, int64_t num_blocks, int dtype, float scale,
               bool fp8, float k_scale, float v_scale, const float* k_scales,
               const float* v_scales, int window, int max_seq_len, int partition_size,
               void* out, void* workspace, int64_t workspace_bytes, void* stream) {
  if (elt_bytes(dtype) == 0) return PA_ERR_DTYPE;
  int st = check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_size,
                              block_size, max_seq_len);
  if (st != PA_OK) return st;
  if (partition_size < 0 || num_blocks < 0 || block_tables_stride < 0) return PA_ERR_SHAPE;
  if (fp8 && (!(k_scale > 0.f) || !(v_scale > 0.f))) return PA_ERR_SHAPE;
  if ((int64_t)max_seq_len > block_tables_stride * block_size) return PA_ERR_OUT_OF_RANGE;
  if (num_seqs == 0) return PA_OK;
  if (!q || !key_cache || !value_cache || !block_tables || !seq_lens || !out)
    return PA_ERR_NULL;
  if (!aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache) || !aligned16(out))
    return PA_ERR_ALIGN;
  int dev;
  st = device_setup(&dev);
  if (st != PA_OK) return st;
  pa::DecodeArgs a;
  a.q = q; a.kc = key_cache; a.vc = value_cache;
  a.tables = block_tables; a.table_stride = block_tables_stride; a.seq_lens = seq_lens;
  a.num_seqs = num_seqs; a.num_q_heads = num_q_heads; a.num_kv_heads = num_kv_heads;
  a.head_size = head_size; a.block_size = block_size; a.num_blocks = num_blocks;
  a.dtype = dtype; a.scale = scale; a.max_seq_len = max_seq_len; a.window = window;
  a.k_scales = k_scales; a.v_scales = v_scales;
  partitioning(num_seqs, num_q_heads, num_kv_heads, block_size,
               covered_len(max_seq_len, window), partition_size, g_sm_count[dev],
               windowed(max_seq_len, window), fp8 && pa::mma_fp8_path_applies(a),
               &a.num_splits, &a.partition);
  // a window cuts every long sequence to about the same work: one wave of
  // tensor-core CTAs walks the items (wave_plan)
  a.items_per_cta = 1;
  a.even_ctas = 0;
  a.ws_acc = nullptr; a.ws_ml = nullptr; a.ws_rec = nullptr;
  const bool tc16 = !fp8 && pa::mma_path_applies(a);
  const bool tc8 = fp8 && pa::mma_fp8_path_applies(a);
  int64_t C = 0;
  if (even_applies(num_seqs, head_size, max_seq_len, window, partition_size, tc16 || tc8))
    wave_plan(num_seqs, num_kv_heads, a.num_splits, max_seq_len, window, g_sm_count[dev],
              tc8 ? 3 : 2, &a.items_per_cta, &C);
  if (C > 0) {
    const int group = num_q_heads / num_kv_heads;
    const int64_t need = even_workspace(C, group, head_size);
    if (!workspace || workspace_bytes < need) return PA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PA_ERR_ALIGN;
    char* w = static_cast<char*>(workspace);
    const int64_t acc = ((C * 2 * group * head_size * 4 + 255) / 256) * 256;
    const int64_t ml = ((C * 2 * group * 2 * 4 + 255) / 256) * 256;
    a.even_ctas = (int)C;
    a.num_splits = 1;
    a.ws_acc = reinterpret_cast<float*>(w);
    a.ws_ml = reinterpret_cast<float*>(w + acc);
    a.ws_rec = reinterpret_cast<int*>(w + acc + ml);
  } else {
    const int64_t need = workspace_for(num_seqs, num_q_heads, head_size, a.num_splits);
    if (need > 0) {
      if (!workspace || workspace_bytes < need) return PA_ERR_WORKSPACE;
      if (!aligned16(workspace)) return PA_ERR_ALIGN;
      const int64_t n = (int64_t)num_seqs * num_q_heads * a.num_splits;
      a.ws_acc = static_cast<float*>(workspace);
      a.ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                         ((n * head_size * 4 + 255) / 256) * 256);
    }
  }
  a.out = out;
  a.err = g_err_ptr[dev];
  cudaStream_t cs = (cudaStream_t)stream;
  return check_launch(fp8 ? pa::launch_decode_fp8(a, k_scale, v_scale, cs)
                          : pa::launch_decode(a, cs));
}

}  // namespace
