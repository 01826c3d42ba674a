// pa_decode_attention_static: paged decode attention for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand the library a scratch buffer: a serving
// engine that reserved nearly all of HBM for its KV block pool at start-up
// and keeps nothing back for per-call buffers, or a host program whose
// allocation policy forbids cudaMalloc on the decode path (cudaMalloc can
// synchronise the device and stall every stream). For them this entry point
// takes its split-partition scratch from a fixed array that lives in the
// library itself, so a call allocates nothing.
//
// The array below is PA_STATIC_SCRATCH_BYTES on every device that loads the
// library and stays reserved until the process exits. Host code must not
// use the array's name as a device address (on the host it names a stand-in,
// not device memory), so the device address is looked up once per device,
// with that device current, and passed to the kernels.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pagedattn.h"

static __device__ __align__(256) unsigned char g_pa_static_scratch[PA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];   // non-null once found for that device
std::mutex g_scratch_mu;

// Device address of this device's copy of the scratch array, looked up with
// the device current on the first call that succeeds. A failed lookup is not
// remembered: the next call tries again.
int scratch_for_current_device(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return PA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_static_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();   // do not leave the failure for the next call to see
      return PA_ERR_DEVICE;
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" int pa_decode_attention_static(
    const void* q, const void* key_cache, const void* value_cache,
    const int32_t* block_tables, int64_t block_tables_stride, const int32_t* seq_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_size, int block_size,
    int64_t num_blocks, int dtype, float scale, int max_seq_len, int partition_size,
    void* out, void* stream) {
  // Size check first: a problem whose partials do not fit is refused before
  // anything is launched.
  const int64_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                 head_size, block_size, max_seq_len,
                                                 partition_size);
  if (need < 0) return (int)need;
  if (need > (int64_t)PA_STATIC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != PA_OK) return st;
  return pa_decode_attention(q, key_cache, value_cache, block_tables, block_tables_stride,
                             seq_lens, num_seqs, num_q_heads, num_kv_heads, head_size,
                             block_size, num_blocks, dtype, scale, max_seq_len,
                             partition_size, out, scratch, (int64_t)PA_STATIC_SCRATCH_BYTES,
                             stream);
}
