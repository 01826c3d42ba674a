/*
 * pagedattn.h — C ABI of libpagedattn.so, the paged-KV decode hot path for
 * NVIDIA GB300 (sm_103a).
 *
 * The method (PagedAttention): a sequence's key/value cache is cut into
 * fixed-size blocks of B tokens that may sit anywhere in a preallocated
 * physical pool; a per-request block table maps logical block i to its
 * physical block, and the attention kernel reads the cache only through that
 * table.  Sources, by page title:
 *   [P1] "PagedAttention 核心创新深度分析" (openeuler.csdn.net)
 *   [P2] "Visual reading: paged-attention-kv-cache" (blog.vllbc.top)
 *   [P3] "vLLM 的 PagedAttention：显存管理如何撑起大模型推理" (deepsonar.com.cn)
 *   [P4] "Infra: PagedAttention" (pufanyi.com)
 *
 * Conventions shared by every call
 *   - All data pointers are DEVICE pointers unless a parameter says "host".
 *     The caller owns every buffer; the library keeps no per-call state and
 *     never allocates device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Every call is asynchronous on that stream; a return of PA_OK
 *     means the arguments were valid and the kernels were launched.
 *   - The decode step's kernels (slot mapping, KV writes, decode attention
 *     and its combine or merge) are launched with programmatic dependent
 *     launch: a kernel's blocks may be scheduled while the kernel before it
 *     in the stream drains, but each waits for that kernel to complete, and
 *     for its writes to be visible, before it touches memory that kernel
 *     or any earlier one may write. Stream order is kept for every caller;
 *     only launch latency and block set-up overlap.
 *   - Tensors are dense row-major in the shapes given below.
 *   - Physical KV pool layout (one pool for K, one for V):
 *         cache[num_blocks][num_kv_heads][block_size][head_size]
 *     A slot id s names block s / block_size, row s % block_size.  Every
 *     (block, kv head) slice is one contiguous run of block_size*head_size
 *     elements.
 *   - dtype codes: PA_F32, PA_F16, PA_BF16. q, k, v, caches and out share
 *     one dtype. Attention arithmetic is fp32.
 *   - Supported shapes: slot mapping and the KV write take any block_size
 *     >= 1 and any head_size whose row is a multiple of 16 bytes. Attention
 *     takes head_size in {64, 128}, block_size a power of two in [1, 256],
 *     and num_q_heads a multiple of num_kv_heads with group size
 *     num_q_heads / num_kv_heads in {1, 2, 4, 8}.
 *   - Device pointers must be 16-byte aligned (PA_ERR_ALIGN otherwise).
 *   - Kernels check every index they read from device memory (block ids,
 *     positions, slots, sequence lengths) before using it. A bad value is
 *     never dereferenced: the affected item is skipped (slot mapping writes
 *     -1; attention writes zeros for a sequence whose length is out of range
 *     and leaves out a token whose block id is outside the pool) and an
 *     error code is latched in a device-side word; read and clear it with
 *     pa_get_device_error().
 */
#ifndef PAGEDATTN_H_
#define PAGEDATTN_H_

#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ----------------------------------------------------- */
#define PA_OK                0
#define PA_ERR_NULL         (-1)  /* a required pointer is NULL */
#define PA_ERR_SHAPE        (-2)  /* unsupported or inconsistent size */
#define PA_ERR_DTYPE        (-3)  /* unknown dtype code */
#define PA_ERR_WORKSPACE    (-4)  /* workspace missing or too small */
#define PA_ERR_OUT_OF_RANGE (-5)  /* an index is outside its array */
#define PA_ERR_CUDA         (-6)  /* a CUDA runtime call or launch failed */
#define PA_ERR_ALIAS        (-7)  /* copy pairs overlap (dst repeated, or dst is a src) */
#define PA_ERR_ALIGN        (-8)  /* a device pointer is not 16-byte aligned */
#define PA_ERR_DEVICE       (-9)  /* no usable sm_103 device / kernel image */
#define PA_ERR_TIMEOUT      (-10) /* a kernel gave up on a stuck asynchronous copy */

/* ---- dtype codes -------------------------------------------------------- */
#define PA_F32  0
#define PA_F16  1
#define PA_BF16 2

/* Human-readable name of a status code (static string, never NULL). */
PA_API const char* pa_status_string(int status);

/* Library ABI version; bumps whenever a signature or layout changes. */
PA_API int pa_abi_version(void);

/*
 * pa_compute_slot_mapping — [P1] §2.3 BlockTable / slot-mapping kernel (the
 * single-rank case: no context parallelism, so every token is local).
 *
 * For every token t of request r, i.e. query_start_loc[r] <= t <
 * query_start_loc[r+1]:
 *     lb = positions[t] / block_size                 (logical block)
 *     slot_mapping[t] = block_table[r*block_table_stride + lb] * block_size
 *                       + positions[t] % block_size
 *
 * query_start_loc    int32 [num_reqs + 1], non-decreasing, device.
 * positions          int64 [num_tokens], device.
 * block_table        int32 [num_reqs][block_table_stride], device; row r
 *                    lists request r's physical block ids in logical order.
 * slot_mapping       int64 [num_tokens], device, written.
 * Tokens that belong to no request get -1 (PAD). A token whose position is
 * negative, whose logical block is >= block_table_stride, or whose table
 * entry is negative also gets -1 and latches PA_ERR_OUT_OF_RANGE on the
 * device.  num_tokens == 0 or num_reqs == 0 is valid (no launch, or all PAD).
 */
PA_API int pa_compute_slot_mapping(const int32_t* query_start_loc, int num_reqs,
                            const int64_t* positions, int64_t num_tokens,
                            const int32_t* block_table,
                            int64_t block_table_stride, int block_size,
                            int64_t* slot_mapping, void* stream);

/*
 * pa_reshape_and_cache — write the new tokens' keys and values into the pool
 * at the slots the slot mapping produced ([P1] §2.3: the slot mapping lets
 * the attention kernel address the pool directly).
 *
 * k, v          [num_tokens][num_kv_heads][head_size], dtype, device.
 * slot_mapping  int64 [num_tokens], device. slot < 0 (PAD) is skipped;
 *               slot >= num_blocks*block_size is skipped and latches
 *               PA_ERR_OUT_OF_RANGE.
 * key_cache, value_cache  the pools (layout above), device, updated in place.
 * Two tokens mapped to the same slot is a caller error (last writer is
 * unspecified).
 */
PA_API int pa_reshape_and_cache(const void* k, const void* v, int64_t num_tokens,
                         int num_kv_heads, int head_size, int dtype,
                         const int64_t* slot_mapping, void* key_cache,
                         void* value_cache, int64_t num_blocks,
                         int block_size, void* stream);

/*
 * Scratch needed by pa_decode_attention for the same arguments
 * (bytes; 0 means no workspace is needed and NULL may be passed).
 * partition_size as in pa_decode_attention. Returns a negative status on
 * invalid sizes.
 */
PA_API int64_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads,
                                  int num_kv_heads, int head_size,
                                  int block_size, int max_seq_len,
                                  int partition_size);

/*
 * Number of context partitions ("splits") pa_decode_attention uses per
 * sequence of length max_seq_len, and the partition length in tokens that
 * it resolves partition_size to. Either output pointer (host) may be NULL.
 */
PA_API int pa_decode_partitioning(int num_seqs, int num_q_heads,
                                  int num_kv_heads, int block_size,
                           int max_seq_len, int partition_size,
                           int* num_splits_out, int* partition_tokens_out);

/*
 * pa_decode_attention — paged decode attention: one query token per sequence
 * attends over that sequence's cached tokens, read block by block through
 * its block table ([P2] block-wise attention and block table section; [P3]
 * §2.2 and §2.6; [P4] "按 Block 分配"). Paging keeps dense semantics ([P4]
 * closing section), so for each sequence s and query head h, with KV head
 * kvh = h / (num_q_heads / num_kv_heads) and L = seq_lens[s]:
 *     x_j = scale * <q[s,h], K_s[j]>          j < L
 *     out[s,h] = sum_j softmax(x)_j * V_s[j]
 * where K_s[j] is row j % B of KV head kvh in physical block
 * block_tables[s*block_tables_stride + j / B].
 *
 * q, out        [num_seqs][num_q_heads][head_size], dtype, device.
 * key_cache, value_cache  pools (layout above), device.
 * block_tables  int32 [num_seqs][block_tables_stride], device.
 * seq_lens      int32 [num_seqs], device; 0 <= seq_lens[s] <= max_seq_len and
 *               <= block_tables_stride*block_size. A length outside that
 *               range latches PA_ERR_OUT_OF_RANGE and yields zeros; a length
 *               of 0 yields zeros (attention over nothing).
 * max_seq_len   host upper bound of seq_lens, used to size the grid.
 * partition_size  tokens per context partition (split-K over block ranges,
 *               with a log-sum-exp combine), rounded up to a multiple of
 *               max(64, block_size); 0 picks a size from the SM count and the
 *               problem shape.
 * workspace     device scratch of pa_decode_workspace_bytes(...) bytes (may
 *               be NULL when that is 0). Contents on entry are ignored.
 * Accumulation is fp32; out is rounded to nearest in the q dtype. Results
 * are bitwise reproducible for fixed arguments and do not depend on where
 * blocks sit in the pool.
 */
PA_API int pa_decode_attention(const void* q, const void* key_cache,
                        const void* value_cache, const int32_t* block_tables,
                        int64_t block_tables_stride, const int32_t* seq_lens,
                        int num_seqs, int num_q_heads, int num_kv_heads,
                        int head_size, int block_size, int64_t num_blocks,
                        int dtype, float scale, int max_seq_len,
                        int partition_size, void* out, void* workspace,
                        int64_t workspace_bytes, void* stream);

/*
 * pa_decode_attention_static — the same computation as pa_decode_attention,
 * for callers that cannot allocate device memory and so cannot pass a
 * workspace: for example a serving engine that reserved almost all of HBM
 * for its KV block pool up front, or a host whose policy forbids cudaMalloc
 * on the decode path (it can synchronise the device). The paper has no
 * counterpart to this call; it is a convenience of this library.
 *
 * Arguments are those of pa_decode_attention without workspace and
 * workspace_bytes. The split-partition scratch comes from a fixed array of
 * PA_STATIC_SCRATCH_BYTES bytes inside the library, present on every device
 * that loads the library until the process exits. The call allocates
 * nothing.
 *   - Sizes whose scratch (pa_decode_workspace_bytes) exceeds
 *     PA_STATIC_SCRATCH_BYTES are refused with PA_ERR_WORKSPACE before any
 *     launch; use pa_decode_attention with your own workspace for those.
 *   - The first call on a device looks up that device's address of the
 *     array (cudaGetSymbolAddress, with the device current); make that
 *     first call before any stream capture. If the lookup fails the call
 *     returns PA_ERR_DEVICE and the next call on that device tries again.
 *   - All calls on a device share the one array and it keeps whatever the
 *     last call left in it (nothing in it needs to start at zero). Calls
 *     that may run at the same time on the GPU (different streams without
 *     ordering between them) race on it: order them on one stream or use
 *     pa_decode_attention with separate workspaces.
 */
#define PA_STATIC_SCRATCH_BYTES (32ll << 20)
PA_API int pa_decode_attention_static(const void* q, const void* key_cache,
                                      const void* value_cache,
                                      const int32_t* block_tables,
                                      int64_t block_tables_stride,
                                      const int32_t* seq_lens, int num_seqs,
                                      int num_q_heads, int num_kv_heads,
                                      int head_size, int block_size,
                                      int64_t num_blocks, int dtype, float scale,
                                      int max_seq_len, int partition_size,
                                      void* out, void* stream);

/*
 * pa_multi_query_attention — causal paged attention for several new tokens
 * per sequence in one step: a prefill chunk or speculative candidates ([P3]
 * §2.5: one token budget per request covers chunked prefill and speculative
 * tokens; [P1] §2.3: the slot mapping places any number of tokens per
 * request). Sequence s has n_s = query_start_loc[s+1] - query_start_loc[s]
 * new tokens whose K/V are already in the pool (pa_reshape_and_cache) and
 * L_s = seq_lens[s] tokens in total; new token i is at position
 * L_s - n_s + i and attends to positions 0 .. L_s - n_s + i:
 *     out[t, h] = sum_{j <= L_s - n_s + i} softmax_j(scale <q[t,h], K_s[j]>) V_s[j]
 * with t = query_start_loc[s] + i and KV head h / (num_q_heads/num_kv_heads).
 * With n_s = 1 this is pa_decode_attention.
 *
 * q, out           [num_tokens][num_q_heads][head_size], dtype, device;
 *                  num_tokens = query_start_loc[num_seqs].
 * query_start_loc  int32 [num_seqs + 1], non-decreasing, device.
 * seq_lens         int32 [num_seqs], device; n_s <= L_s <= max_seq_len.
 * max_query_len    host upper bound of n_s (sizes the grid).
 * num_tokens       host: rows of q (= query_start_loc[num_seqs]).
 * partition_size   tokens per KV partition (split-K with a log-sum-exp
 *                  combine); 0 splits only short query runs (every
 *                  sequence's rows fit one 64-row tile), sized from the SM
 *                  count. workspace as sized by pa_multi_query_workspace_bytes.
 * Other arguments as in pa_decode_attention. Supported: fp16/bf16,
 * head_size 64/128, block_size a power of two in [8, 256], group size
 * 1/2/4/8 (PA_ERR_SHAPE / PA_ERR_DTYPE otherwise). A sequence whose lengths
 * break these bounds is skipped (its rows are not written) and latches
 * PA_ERR_OUT_OF_RANGE.
 */
PA_API int pa_multi_query_attention(const void* q, const int32_t* query_start_loc,
                                    int num_seqs, int64_t num_tokens,
                                    const void* key_cache, const void* value_cache,
                                    const int32_t* block_tables,
                                    int64_t block_tables_stride, const int32_t* seq_lens,
                                    int num_q_heads, int num_kv_heads, int head_size,
                                    int block_size, int64_t num_blocks, int dtype,
                                    float scale, int max_query_len, int max_seq_len,
                                    int partition_size, void* out, void* workspace,
                                    int64_t workspace_bytes, void* stream);

/*
 * Scratch bytes pa_multi_query_attention needs for these sizes (0: none,
 * NULL may be passed); negative status on invalid sizes.
 */
PA_API int64_t pa_multi_query_workspace_bytes(int64_t num_tokens, int num_seqs,
                                              int num_q_heads, int num_kv_heads,
                                              int head_size, int block_size,
                                              int max_query_len, int max_seq_len,
                                              int partition_size);

/*
 * fp8 KV pools ([P1] §3.5: an attention layer's KV spec carries a
 * quantisation mode; §7 outlook: quantisation-aware blocks). The pages fix no
 * format; this library stores OCP FP8 E4M3 codes (1 byte, same pool layout)
 * with one fp32 scale per pool:
 *     code  = e4m3(x / scale)   nearest even, saturated to +-448, NaN -> NaN
 *     value = code * scale
 *
 * pa_reshape_and_cache_fp8 — pa_reshape_and_cache into fp8 pools: k, v of
 * `dtype` (fp32/fp16/bf16) are divided by k_scale / v_scale in fp32 and
 * converted; head_size a multiple of 16; scales > 0.
 */
PA_API int pa_reshape_and_cache_fp8(const void* k, const void* v, int64_t num_tokens,
                                    int num_kv_heads, int head_size, int dtype,
                                    const int64_t* slot_mapping, void* key_cache,
                                    void* value_cache, int64_t num_blocks, int block_size,
                                    float k_scale, float v_scale, void* stream);

/*
 * pa_decode_attention_fp8 — pa_decode_attention over fp8 pools: q and out of
 * `dtype`, K = code * k_scale, V = code * v_scale. The workspace is sized by
 * pa_decode_fp8_workspace_bytes with the same arguments (window 0). The
 * partitioning differs from pa_decode_attention's: 16-bit queries, head size
 * 128 and blocks of at least 8 tokens run the tensor-core kernel, which
 * takes the tensor-core partition sizes for every group size and, for a
 * window that cuts the longest sequence, one wave of three CTAs per SM
 * (pa_decode_even_ctas). pa_decode_fp8_partitioning reports the
 * partitions. k_scale and v_scale must be positive (else PA_ERR_SHAPE).
 */
/*
 * pa_decode_fp8_workspace_bytes — scratch for the fp8-pool decode calls
 * (pa_decode_attention_fp8 with window 0, pa_decode_attention_fp8_window,
 * pa_decode_attention_fp8_scaled) with the same arguments; dtype is the
 * query type. Negative status on invalid sizes.
 */
PA_API int64_t pa_decode_fp8_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                             int head_size, int block_size, int dtype,
                                             int max_seq_len, int window, int partition_size);
PA_API int pa_decode_attention_fp8(const void* q, const void* key_cache,
                                   const void* value_cache, const int32_t* block_tables,
                                   int64_t block_tables_stride, const int32_t* seq_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads,
                                   int head_size, int block_size, int64_t num_blocks,
                                   int dtype, float scale, float k_scale, float v_scale,
                                   int max_seq_len, int partition_size, void* out,
                                   void* workspace, int64_t workspace_bytes, void* stream);

/*
 * fp8 blocks that carry their own scales ([P1] §3.5 kv_quant_mode and §7.4,
 * the compression-aware block: the quantisation belongs to the block). The
 * same E4M3 pools as above, plus two fp32 arrays k_scales, v_scales
 * [num_blocks][num_kv_heads] (device, caller-owned, 16-byte aligned): the
 * scale of (block b, KV head h) is a power of two,
 *     value = code * scales[b][h].
 * Reading taken (the pages fix no format): a block's scales are fixed by
 * the KV write that stores its first row (row 0). That write takes the
 * token landing there and the tokens right after it in the same call whose
 * slots continue it inside the block (a prefill chunk fills up to
 * block_size rows at once; a decode step writes one), and from the largest
 * |value| amax among them (per head, K and V separately; NaN left out) sets
 *     scale = 2^k,  k = ceil(log2(amax)) - 7 kept in [-126, 127]
 *     (amax = 0 gives 1),
 * so those tokens' largest magnitude lands in (64, 128] and later tokens of
 * the block have 3.5x headroom before the largest code (448) saturates. Every
 * token of the call is then quantised with its block's scale, as in
 * pa_reshape_and_cache_fp8 (IEEE fp32 division, nearest even, saturated).
 * Blocks whose first row the call does not write keep their scales. When a
 * block is copied for copy-on-write, copy its scales with it: pa_copy_blocks
 * on the scale arrays with block_bytes = num_kv_heads * 4.
 *
 * pa_reshape_and_cache_fp8_scaled — the write above: two launches on
 * `stream` (the scales of the blocks begun in this call, then the codes).
 * Arguments as in pa_reshape_and_cache_fp8, with k_scales / v_scales in
 * place of the pool scales. Slots out of the pool are skipped and latch
 * PA_ERR_OUT_OF_RANGE; two tokens of a call mapped to one slot are a caller
 * error.
 *
 * pa_decode_attention_fp8_scaled — decode attention over such pools:
 * K_s[j] = code * k_scales[b][h], V_s[j] = code * v_scales[b][h] for the
 * block b holding token j. `window` as in pa_decode_attention_fp8_window
 * (0 = the whole sequence); workspace sized by
 * pa_decode_fp8_workspace_bytes with the same arguments; partitioning as
 * pa_decode_fp8_partitioning reports. The tensor-core kernel multiplies each
 * token's softmax weight by its block's V scale relative to the first
 * attended block's before rounding it to fp16, so V scales within one
 * sequence more than 2^16 apart saturate that weight (a precision limit, not
 * an error).
 */
PA_API int pa_reshape_and_cache_fp8_scaled(const void* k, const void* v, int64_t num_tokens,
                                           int num_kv_heads, int head_size, int dtype,
                                           const int64_t* slot_mapping, void* key_cache,
                                           void* value_cache, float* k_scales,
                                           float* v_scales, int64_t num_blocks,
                                           int block_size, void* stream);
PA_API int pa_decode_attention_fp8_scaled(const void* q, const void* key_cache,
                                          const void* value_cache, const float* k_scales,
                                          const float* v_scales, const int32_t* block_tables,
                                          int64_t block_tables_stride,
                                          const int32_t* seq_lens, int num_seqs,
                                          int num_q_heads, int num_kv_heads, int head_size,
                                          int block_size, int64_t num_blocks, int dtype,
                                          float scale, int window, int max_seq_len,
                                          int partition_size, void* out, void* workspace,
                                          int64_t workspace_bytes, void* stream);

/*
 * Sliding-window decode. The pages name the window through the blocks the
 * allocator may release ("PagedAttention 核心创新深度分析" §3.2
 * allocate_slots, phase 1, and §3.3.1 get_num_blocks_to_allocate: skipped
 * blocks = skipped tokens / block_size). Reading: the query of sequence s
 * attends its last `window` tokens, the new token included:
 *     lo = L - window  if 0 < window < L,  else 0
 *     out[s,h] = sum_{lo <= j < L} softmax(x)_j * V_s[j]
 * window = 0 is plain pa_decode_attention. The table entries of the leading
 * lo / block_size blocks are never read: the caller may have released those
 * blocks and left any value there (e.g. -1).
 *
 * pa_decode_window_workspace_bytes — scratch for pa_decode_attention_window
 * with the same arguments (window >= 0; returns a negative status on
 * invalid sizes).
 * pa_decode_attention_window — pa_decode_attention with a window.
 * pa_decode_attention_fp8_window — pa_decode_attention_fp8 with a window;
 * its scratch comes from pa_decode_fp8_workspace_bytes.
 * Other arguments, layouts and errors as in the unwindowed calls; window < 0
 * is PA_ERR_SHAPE.
 */
/*
 * pa_decode_window_partitioning — pa_decode_partitioning for the windowed
 * calls with the same arguments. When 0 < window < max_seq_len every
 * sequence at least window long covers window .. window + 63 tokens (the
 * window's first tile is read whole), so with partition_size == 0 the
 * partitions are sized for one wave of resident CTAs (the most splits per
 * (sequence, KV head) pair that still fit, at least 256 tokens each) rather
 * than the two waves of the unwindowed calls. Calls for which
 * pa_decode_even_ctas returns a positive count do not use these partitions.
 * window < 0 is PA_ERR_SHAPE.
 *
 * pa_decode_even_ctas — whether a decode call with these sizes runs the
 * even schedule, and over how many CTAs. Calls with a window that cuts the
 * longest sequence (0 < window < max_seq_len), partition_size == 0, head
 * size 128, at most 8192 sequences and the tensor-core kernel (16-bit
 * queries; 16-bit pools with groups of 2, 4 or 8, or fp8 pools with any
 * group; blocks of at least 8 tokens) run one wave of CTAs (SMs x 2 for
 * 16-bit pools, x 3 for fp8 pools). Each CTA takes whole partitions of the fixed partitioning in
 * turn, unless whole partitions would leave the busiest CTA more than 1.25
 * times the mean work; then the even schedule runs: the batch's 64-token
 * tiles — those of every (sequence, KV head) pair in order, each pair from
 * its window's first tile — are cut into C runs of equal length, one per
 * CTA (C = the wave, fewer for small batches), and a second launch merges
 * the pairs cut between CTAs and writes the zero outputs of empty
 * sequences. Returns C (> 0) for such calls, 0 for calls that use the fixed
 * partitions, a negative status on invalid sizes. kv_format: 0 = 16-bit
 * pools, 1 = fp8 pools with one scale per pool, 2 = fp8 pools with
 * per-block scales; dtype is the query type. The workspace queries size
 * the scratch for either schedule.
 */
PA_API int pa_decode_even_ctas(int num_seqs, int num_q_heads, int num_kv_heads, int head_size,
                               int block_size, int dtype, int kv_format, int max_seq_len,
                               int window, int partition_size);
PA_API int pa_decode_window_partitioning(int num_seqs, int num_q_heads, int num_kv_heads,
                                         int block_size, int max_seq_len, int window,
                                         int partition_size, int* num_splits_out,
                                         int* partition_tokens_out);
/*
 * pa_decode_fp8_partitioning — the partition count and length that
 * pa_decode_attention_fp8 (window = 0) or pa_decode_attention_fp8_window
 * uses with the same sizes, unless pa_decode_even_ctas reports the even
 * schedule for them; head_size and dtype (the query type) select the
 * kernel. Either output pointer (host) may be NULL. Invalid sizes give
 * PA_ERR_SHAPE, an unknown dtype PA_ERR_DTYPE.
 */
PA_API int pa_decode_fp8_partitioning(int num_seqs, int num_q_heads, int num_kv_heads,
                                      int head_size, int block_size, int dtype,
                                      int max_seq_len, int window, int partition_size,
                                      int* num_splits_out, int* partition_tokens_out);
PA_API int64_t pa_decode_window_workspace_bytes(int num_seqs, int num_q_heads,
                                                int num_kv_heads, int head_size,
                                                int block_size, int max_seq_len, int window,
                                                int partition_size);
PA_API int pa_decode_attention_window(const void* q, const void* key_cache,
                                      const void* value_cache, const int32_t* block_tables,
                                      int64_t block_tables_stride, const int32_t* seq_lens,
                                      int num_seqs, int num_q_heads, int num_kv_heads,
                                      int head_size, int block_size, int64_t num_blocks,
                                      int dtype, float scale, int window, int max_seq_len,
                                      int partition_size, void* out, void* workspace,
                                      int64_t workspace_bytes, void* stream);
PA_API int pa_decode_attention_fp8_window(const void* q, const void* key_cache,
                                          const void* value_cache,
                                          const int32_t* block_tables,
                                          int64_t block_tables_stride,
                                          const int32_t* seq_lens, int num_seqs,
                                          int num_q_heads, int num_kv_heads, int head_size,
                                          int block_size, int64_t num_blocks, int dtype,
                                          float scale, float k_scale, float v_scale,
                                          int window, int max_seq_len, int partition_size,
                                          void* out, void* workspace,
                                          int64_t workspace_bytes, void* stream);

/*
 * pa_copy_blocks — block-level copy-on-write data movement ([P2] Figure 8,
 * the copy of the shared last block when one sharer diverges; [P4]
 * copy-on-write figure). For every pair (src, dst) in src_dst_pairs and
 * every layer l, the whole K block src of key_caches[l] is copied to block
 * dst, and likewise for value_caches[l].
 *
 * key_caches, value_caches  HOST arrays of num_layers device pointers, one
 *               pool per layer, each [num_blocks][...] with block_bytes bytes
 *               per block (num_kv_heads*block_size*head_size*elt).
 * src_dst_pairs int64 [num_pairs][2], device.
 * src_dst_pairs_host  optional HOST copy of the same pairs (may be NULL). When
 *               given, ids are range-checked and aliasing (a repeated dst, or
 *               a dst that is also a src) is rejected with PA_ERR_ALIAS before
 *               anything is launched. Without it the kernel range-checks each
 *               pair (skipping and latching PA_ERR_OUT_OF_RANGE) and aliasing
 *               is the caller's responsibility.
 * block_bytes   a positive multiple of 4 (16-byte vectors are moved when it
 *               is a multiple of 16, 4-byte words otherwise, e.g. the
 *               per-block scale arrays of fp8 pools: num_kv_heads * 4).
 */
PA_API int pa_copy_blocks(void* const* key_caches, void* const* value_caches,
                   int num_layers, const int64_t* src_dst_pairs,
                   const int64_t* src_dst_pairs_host, int64_t num_pairs,
                   int64_t num_blocks, int64_t block_bytes, void* stream);

/*
 * pa_map_to_kernel_blocks — hybrid block sizes ([P1] §3.4,
 * map_to_kernel_blocks): when the allocator's block holds r kernel blocks,
 * its block k owns kernel blocks k*r, k*r+1, ..., k*r+r-1, and a table of
 * allocator ids expands to a table the attention kernels read with block
 * size B = allocator block tokens / r. Example from [P1]: ids [0, 1, 2] with
 * r = 2 give [0, 1, 2, 3, 4, 5].
 *
 * manager_table  int32 [num_rows][manager_stride], device; the first
 *                num_cols entries of each row are expanded; a negative id
 *                expands to r entries of -1.
 * kernel_table   int32 [num_rows][kernel_stride], device, written in its
 *                first num_cols*r entries of each row;
 *                kernel_stride >= num_cols * r.
 * blocks_per_kv_block  r >= 1. An expanded id above INT32_MAX is written as
 *                -1 and latches PA_ERR_OUT_OF_RANGE.
 */
PA_API int pa_map_to_kernel_blocks(const int32_t* manager_table, int64_t num_rows,
                                   int64_t manager_stride, int64_t num_cols,
                                   int blocks_per_kv_block, int32_t* kernel_table,
                                   int64_t kernel_stride, void* stream);

/*
 * pa_selftest_bounded_wait — exercises the bounded mbarrier wait that every
 * asynchronous kernel of this library relies on (no counterpart on the
 * pages; a failure-detection check). One CTA waits on a barrier phase that
 * nothing completes: warp 0 with a limit of timeout_cycles SM clocks, warp 1
 * with a 1000x longer one. Warp 0 must give up and raise the CTA's abort
 * flag, and warp 1 must leave through that flag. The kernel writes, to the
 * caller's device buffer status[3] (int32): status[0], status[1] =
 * PA_ERR_TIMEOUT for each warp that gave up (PA_OK if its wait completed),
 * status[2] = the abort flag (1). Nothing faults and both waits end by
 * themselves; the context stays usable. 0 < timeout_cycles <= 2^40/1000,
 * else PA_ERR_SHAPE; NULL status is PA_ERR_NULL. Asynchronous on stream.
 */
PA_API int pa_selftest_bounded_wait(int* status, long long timeout_cycles, void* stream);

/*
 * Read (and clear) the device-side error word that the kernels latch on bad
 * indices. Synchronises `stream` first. *code_out receives PA_OK or the
 * first latched error (PA_ERR_OUT_OF_RANGE). The word is per device and
 * shared by all streams.
 */
PA_API int pa_get_device_error(int* code_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H_ */
