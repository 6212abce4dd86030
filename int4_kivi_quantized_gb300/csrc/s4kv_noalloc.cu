// s4kv_decode_attention_noalloc: decode attention whose scratch lives in a
// fixed array compiled into this library, for callers that cannot allocate
// device memory at the point of the call (see include/s4kv.h).

#include "s4kv_common.cuh"

#include <mutex>

namespace {

// The decode kernel's per-warp partial results. Every GPU that loads the
// library holds this array until the process exits. Its contents carry over
// from call to call; the kernel writes each partial before reading it, so
// nothing in it has to start at zero.
static __device__ __align__(256) unsigned char s4kv_noalloc_scratch[S4KV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_lock;
void* g_scratch[kMaxDevices] = {};

// Device address of the array on the cache's device, looked up once per device
// (the host-side name of a __device__ array is not a device address). The
// cache's device must be the current one: the array is reached through the
// current device's copy of the module, and the kernel runs there.
int scratch_for(const s4kv_cache* cache, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return S4KV_ERR_CUDA;
  if (dev != cache->device) return S4KV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> guard(g_lock);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, s4kv_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return S4KV_ERR_CUDA;
    }
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return S4KV_OK;
}

}  // namespace

extern "C" int s4kv_decode_attention_noalloc(s4kv_cache* cache, int layer, const void* q, int num_q_heads,
                                             const int32_t* block_table, int bt_stride,
                                             const int32_t* seq_lens, const int32_t* slot_ids, int B,
                                             float sm_scale, void* out, int out_dtype, int max_seq_len,
                                             void* stream) {
  if (!cache) return S4KV_ERR_INVALID_ARG;
  size_t need = 0;
  const int rc = s4kv_decode_workspace_bytes(cache, B, num_q_heads, max_seq_len, &need);
  if (rc != S4KV_OK) return rc;
  if (need > S4KV_NOALLOC_SCRATCH_BYTES) return S4KV_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const int rs = scratch_for(cache, &scratch);
  if (rs != S4KV_OK) return rs;
  return s4kv_decode_attention(cache, layer, q, num_q_heads, block_table, bt_stride, seq_lens, slot_ids, B,
                               sm_scale, out, out_dtype, scratch, S4KV_NOALLOC_SCRATCH_BYTES, max_seq_len,
                               stream);
}
