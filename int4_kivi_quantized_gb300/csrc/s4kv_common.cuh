// Internal definitions shared by the s4kv CUDA translation units (not part of
// the public ABI; see include/s4kv.h for the format and the calls).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "../../include/s4kv.h"

namespace s4kv {

// Fixed geometry of the one supported configuration.
constexpr int kD = 128;          // head_dim
constexpr int kP = 16;           // tokens per page
constexpr int kG = 32;           // tokens per key group
constexpr int kGv = 32;          // channels per value group
// Record of one (page, kv head): key codes, key scale/min, value codes, value
// scale/min (fp32). 4-bit codes: 3072 bytes; 2-bit codes: 2048 bytes.
template <int BITS>
struct Rec {
  static_assert(BITS == 4 || BITS == 2, "4-bit or 2-bit codes");
  static constexpr int kBytes = BITS == 4 ? 3072 : 2048;
  static constexpr int kKc = 0;
  static constexpr int kKm = 256 * BITS;              // key codes: 16 tokens x 128 channels x BITS bits
  static constexpr int kVc = kKm + 512;
  static constexpr int kVm = kVc + 256 * BITS;
  static constexpr int kLevels = (1 << BITS) - 1;     // largest code
  static_assert(kVm + 512 == kBytes, "four regions fill the record");
};
// FP8 E4M3 record (bits = 8): 4096 bytes, key bytes then value bytes, one e4m3
// byte per element and no per-group metadata (one scale per layer, kv head and
// tensor, kept in the pool header).
template <>
struct Rec<8> {
  static constexpr int kBytes = 4096;
  static constexpr int kKc = 0;
  static constexpr int kVc = 2048;
};
constexpr int kRec = Rec<4>::kBytes;
constexpr int kKc = Rec<4>::kKc, kKm = Rec<4>::kKm, kVc = Rec<4>::kVc, kVm = Rec<4>::kVm;
inline int rec_bytes(int bits) {
  return bits == 2 ? Rec<2>::kBytes : bits == 8 ? Rec<8>::kBytes : Rec<4>::kBytes;
}
constexpr int kMaxGroup = 8;     // largest GQA group (query heads per kv head)

// Status area at the start of the pool (int32 words): the first error, and the
// grid barrier of the decode step (arrival count, generation).
enum { ST_CODE = 0, ST_DETAIL = 1, ST_ARG = 2, ST_BAR_COUNT = 16, ST_BAR_GEN = 17 };

}  // namespace s4kv

struct s4kv_cache {
  s4kv_config cfg;
  char* pool;
  size_t pool_bytes;
  s4kv_layout lay;
  size_t counters_offset;   // int32 [max_slots][H_kv], reserved (no kernel uses it)
  int elem_bytes;
  int decode_warps;         // 0 = every warp of the grid
  int tail_cost;            // cost of a tail chunk in the decode work partition
  int decode_impl;          // 0 tensor-core, 1 FFMA
  int key_split;            // S4KV_OPT_KEY_SPLIT
  int mq_kernel;            // S4KV_OPT_MQ_KERNEL
  int bits;                 // code width of the pages: 4, 2, or 8 (FP8 E4M3)
  long long wait_ns;
  int num_sms;
  int device;
};

namespace s4kv {

struct AppendArgs {
  char* pages;              // layer page region
  char* kring;              // layer key ring region
  char* vring;              // layer value ring region
  int* lens;                // [max_slots][H] stored lengths of this layer
  int* status;
  const uint16_t* k;
  const uint16_t* v;
  const int* cu_new;
  const int* slot_ids;
  const int* seq_lens_before;
  const int* block_table;
  long long kring_slot, kring_head;   // element strides
  long long vring_slot, vring_head;
  int bt_stride, n, num_new, H, R, num_pages, max_slots, dtype;
  int bits;                 // code width: 4, 2 or 8 (FP8)
  const float* fp8_scale;   // FP8: this layer's scales, key [H] then value [H]
};

struct DequantArgs {
  const char* pages;
  const char* kring;
  const char* vring;
  const int* lens;
  int* status;
  const int* bt_row;
  float* out_k;
  float* out_v;
  long long kring_slot, kring_head, vring_slot, vring_head;
  int slot, T, H, R, num_pages, max_slots, dtype;
  int bits;                 // code width: 4, 2 or 8 (FP8)
  const float* fp8_scale;   // FP8: this layer's scales, key [H] then value [H]
};

struct DecodeArgs {
  const char* pages;
  const char* kring;
  const char* vring;
  const int* lens;          // [max_slots][H] stored lengths of this layer
  int* status;
  const uint16_t* q;
  const int* block_table;
  const int* seq_lens;
  const int* slot_ids;
  void* out;
  float* ws;                // two partials per warp, then the partition record
  long long kring_slot, kring_head, vring_slot, vring_head;
  long long wait_ns;
  float sm_scale_log2;      // sm_scale * log2(e)
  int bt_stride, B, Hq, H, g, R, num_pages, max_slots, dtype, out_dtype;
  int max_warps;            // 0: every warp of the grid
  int tail_cost;            // work-partition cost of a tail chunk (key group = 1)
  int max_seq_len;
  int grid_warps;           // worker warps of the launch grid (sizes the partial area)
  int nq;                   // query tokens per sequence (multi-query path; 1 for decode)
  int tw;                   // warps per team (multi-query path): ceil(nq g / 8)
  int pcols;                // columns of one partial in the workspace: g (decode), 8 (multi-query)
  int key_split;            // decode main loop: low f16 part of q' on wide-scale key slices
  int mq_kernel;            // multi-query kernel choice (S4KV_OPT_MQ_KERNEL)
  int bits;                 // code width: 4, 2 or 8 (FP8)
  const float* fp8_scale;   // FP8: this layer's scales, key [H] then value [H]
  // decode step (s4kv_decode_step): the new key and value rows [B][H][128] of
  // the token each sequence appends before attending; null for attention only
  const uint16_t* knew;
  const uint16_t* vnew;
  int* lens_w;              // the stored lengths, written by the step
  unsigned* gbar;           // grid barrier words (arrivals, generation)
};

// Asks for the largest shared-memory carve-out for `func`, once per device and
// kernel: every kernel of the library then runs with the same L1/shared split, so
// an SM needs no reconfiguration between back-to-back launches of different
// kernels (decode, merge, append).
inline cudaError_t prefer_max_shared(const void* func) {
  constexpr int kMax = 256;
  static std::mutex lock;
  static int dev_of[kMax];
  static const void* fn_of[kMax];
  static int n = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return cudaErrorInvalidDevice;
  }
  std::lock_guard<std::mutex> guard(lock);
  for (int i = 0; i < n; ++i)
    if (dev_of[i] == dev && fn_of[i] == func) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e;
  }
  if (n < kMax) {
    dev_of[n] = dev;
    fn_of[n] = func;
    ++n;
  }
  return cudaSuccess;
}

// Host-side launchers (one per translation unit).
cudaError_t launch_append(const AppendArgs& a, int grid, cudaStream_t st);
int append_ctas_per_sm();   // resident CTAs per SM the append kernel is sized for
cudaError_t launch_dequant(const DequantArgs& a, cudaStream_t st);
cudaError_t launch_decode(const DecodeArgs& a, int impl, int grid, cudaStream_t st);
// the decode step: a cooperative launch of the decode kernel with the append phase
cudaError_t launch_decode_step(const DecodeArgs& a, int impl, int grid, cudaStream_t st);
cudaError_t launch_mq(const DecodeArgs& a, int grid, cudaStream_t st);
int decode_threads(int impl);
int decode_warps_per_cta(int impl);
size_t decode_partial_bytes(int g);
size_t decode_meta_bytes(int B, int H);   // merge descriptors, one per (sequence, kv head)
size_t decode_trace_bytes_per_warp();   // 0 unless built with -DS4KV_DECODE_TRACE
size_t decode_smem_bytes(int impl, int B);
int decode_ctas_per_sm(int impl, int B);

// ---- device helpers ----------------------------------------------------------
__device__ __forceinline__ void report(int* status, int code, int detail, int arg) {
  if (atomicCAS(status + ST_CODE, 0, code) == 0) {
    status[ST_DETAIL] = detail;
    status[ST_ARG] = arg;
  }
}

__device__ __forceinline__ float widen16(uint16_t bits, int dtype) {
  if (dtype == S4KV_BF16) return __uint_as_float(static_cast<uint32_t>(bits) << 16);
  return __half2float(__ushort_as_half(bits));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

}  // namespace s4kv
