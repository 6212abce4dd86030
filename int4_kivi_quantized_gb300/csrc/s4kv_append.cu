// Write side of the cache: quantize-on-write with residual flush (s4kv_append),
// and the exact restore used for byte-level checks (s4kv_dequant_debug).
//
// Method ("4.4 KV Cache 量化", sections 3.1 and 3.2): a key group is G = 32
// consecutive tokens of one channel; a value group is Gv = 32 channels of one
// token; each group keeps fp32 (scale, min) and 4-bit codes from the min/max
// asymmetric mapping. New key tokens wait in the key ring until their group is
// complete; values stay in a window of the newest R tokens and are quantized
// as they leave it. "给 KV cache 减肥" section 3.1: quantize before the write.
//
// This translation unit is compiled with -fmad=false and spells every rounding
// out (__fsub_rn, __fdiv_rn, __float2int_rn, __fmaf_rn) so that codes and
// metadata are bit-identical to the IEEE definition of the quantizer.

#include "s4kv_common.cuh"

#include <cuda_fp8.h>
#include <climits>

namespace s4kv {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxSeqsPerCall = 8192;

__device__ __forceinline__ const uint16_t* row_ptr(const uint16_t* base, long long row, int H, int h) {
  return base + (row * H + h) * kD;
}

// Range of 32-token tiles of new tokens that need quantizing straight from the
// input: key groups made only of new tokens, and value tokens that are already
// outside the window when the append ends. Returns the count, sets *lo.
__device__ __forceinline__ int tile_range(int T0, int T1, int R, int* lo) {
  const int Tk1 = T1 & ~(kG - 1);
  const int Tv1 = max(0, T1 - R);
  const int kA = (T0 + kG - 1) / kG, kB = Tk1 / kG;
  int l = INT_MAX, h = INT_MIN;
  if (kB > kA) { l = kA; h = kB; }
  if (Tv1 > T0) {
    l = min(l, T0 / 32);
    h = max(h, (Tv1 + 31) / 32);
  }
  *lo = l;
  return h > l ? h - l : 0;
}

// Exact quantization of one value x given the group's (lo, s): codes 0 .. 2^BITS - 1.
template <int BITS>
__device__ __forceinline__ int quant_code(float x, float lo, float s) {
  if (s == 0.0f) return 0;
  int c = __float2int_rn(__fdiv_rn(__fsub_rn(x, lo), s));
  return min(max(c, 0), Rec<BITS>::kLevels);
}

struct Ctx {
  const AppendArgs* a;
  const int* bt_row;
  int slot;
};

template <int BITS>
__device__ __forceinline__ char* record(const Ctx& c, int logical_page, int h) {
  const int pp = c.bt_row[logical_page];
  if (pp < 0 || pp >= c.a->num_pages) {
    report(c.a->status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp);
    return nullptr;
  }
  return c.a->pages + (static_cast<long long>(pp) * c.a->H + h) * Rec<BITS>::kBytes;
}

// Quantizes key group `grp` of head h (32 tokens x 128 channels) whose token
// rows are src[0..31], and writes the two pages' key codes and metadata.
// Each lane owns one channel and walks down the 32 tokens (a per-channel group).
// 2-bit codes: a byte holds the codes of channel slices kk and kk + 1 (lanes 4
// apart), so the even slice's lane fetches its partner's codes and writes it.
// Called by all 128 threads.
template <int BITS>
__device__ void key_flush(const Ctx& c, int h, int grp, const uint16_t* const* src,
                          uint8_t (*stage)[1536]) {
  using F = Rec<BITS>;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int ch = 32 * w + lane;
  float x[kG];
  float lo, hi;
#pragma unroll
  for (int t = 0; t < kG; ++t) x[t] = widen16(src[t][ch], c.a->dtype);
  lo = x[0];
  hi = x[0];
#pragma unroll
  for (int t = 1; t < kG; ++t) {
    lo = fminf(lo, x[t]);
    hi = fmaxf(hi, x[t]);
  }
  lo = __fadd_rn(lo, 0.0f);
  hi = __fadd_rn(hi, 0.0f);
  const float s = __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(F::kLevels));
  const int kk = lane >> 2, j = lane & 3;
  const int bj = (j == 0) ? 0 : (j == 1) ? 2 : (j == 2) ? 1 : 3;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
#pragma unroll
    for (int a = 0; a < 8; ++a) {
      const int lo_c = quant_code<BITS>(x[16 * p + a], lo, s);
      const int hi_c = quant_code<BITS>(x[16 * p + a + 8], lo, s);
      if constexpr (BITS == 4) {
        stage[p][(kk >> 2) * 512 + (4 * a + w) * 16 + (kk & 3) * 4 + bj] =
            static_cast<uint8_t>(lo_c | (hi_c << 4));
      } else {
        const int mine = lo_c | (hi_c << 2);                        // positions 0, 1 (or 2, 3)
        const int other = __shfl_xor_sync(0xffffffffu, mine, 4);   // the odd slice's lane
        if ((kk & 1) == 0)
          stage[p][(4 * a + w) * 16 + (kk >> 1) * 4 + bj] = static_cast<uint8_t>(mine | (other << 4));
      }
    }
  }
  {
    const int p = w >> 1, u = w & 1, i = lane >> 2, e = lane & 3;
    float* meta = reinterpret_cast<float*>(stage[p] + F::kKm);
    meta[((2 * i + u) * 16 + 4 * e) / 4] = s;
    meta[((2 * i + u) * 16 + 4 * e + 256) / 4] = lo;
  }
  __syncthreads();
  constexpr int kChunks = (F::kKm + 512) / 16;   // key codes and key metadata of one page
  for (int q = tid; q < 2 * kChunks; q += kThreads) {
    const int p = q / kChunks, off = (q % kChunks) * 16;
    char* rec = record<BITS>(c, 2 * grp + p, h);
    if (rec) *reinterpret_cast<uint4*>(rec + off) = *reinterpret_cast<const uint4*>(stage[p] + off);
  }
  __syncthreads();
}

// Quantizes one value token (absolute position t) of head h from row `src`
// and writes its codes and metadata into its page slot. One warp; lane l owns
// channels 4l..4l+3 and the 8 lanes of a 32-channel group reduce by shuffles.
template <int BITS>
__device__ void value_token_row(const Ctx& c, int h, int t, uint2 raw, int pp);

template <int BITS>
__device__ void value_token(const Ctx& c, int h, int t, const uint16_t* src) {
  const int l = threadIdx.x & 31;
  value_token_row<BITS>(c, h, t, *reinterpret_cast<const uint2*>(src + 4 * l), c.bt_row[t / kP]);
}

// The same, with this lane's four values (raw) and the token's pool page (pp)
// already loaded.
template <int BITS>
__device__ void value_token_row(const Ctx& c, int h, int t, uint2 raw, int pp) {
  using F = Rec<BITS>;
  const int l = threadIdx.x & 31;
  float x[4];
  x[0] = widen16(static_cast<uint16_t>(raw.x & 0xffff), c.a->dtype);
  x[1] = widen16(static_cast<uint16_t>(raw.x >> 16), c.a->dtype);
  x[2] = widen16(static_cast<uint16_t>(raw.y & 0xffff), c.a->dtype);
  x[3] = widen16(static_cast<uint16_t>(raw.y >> 16), c.a->dtype);
  float lo = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
  float hi = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, m));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, m));
  }
  lo = __fadd_rn(lo, 0.0f);
  hi = __fadd_rn(hi, 0.0f);
  const float s = __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(F::kLevels));
  int c4 = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) c4 |= quant_code<BITS>(x[q], lo, s) << (4 * q);
  const int partner = __shfl_down_sync(0xffffffffu, c4, 2);
  // 2-bit: lane (mp, a) = 8 mp + a gathers the byte of channels 32 mp + 8 q + a
  // (q = 0..3), held by lanes 8 mp + 2 q + a / 4 as element a % 4
  int crumbs = 0;
  if constexpr (BITS == 2) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int v = __shfl_sync(0xffffffffu, c4, 8 * (l >> 3) + 2 * q + ((l & 7) >> 2));
      crumbs |= ((v >> (4 * (l & 3))) & 3) << (2 * q);
    }
  }
  if (pp < 0 || pp >= c.a->num_pages) {
    if (l == 0) report(c.a->status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp);
    return;
  }
  char* rec = c.a->pages + (static_cast<long long>(pp) * c.a->H + h) * F::kBytes;
  const int tau = t % kP;
  const int b = (tau & 7) >> 1, wv = tau >> 3, r = tau & 1;
  const int bt = wv ? (r ? 3 : 1) : (r ? 2 : 0);
  const int e = r + 2 * wv;
  if constexpr (BITS == 4) {
    if ((l & 3) < 2) {
      const int mt = l >> 2;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int a = 4 * (l & 1) + q;
        const int byte = ((c4 >> (4 * q)) & 15) | (((partner >> (4 * q)) & 15) << 4);
        rec[F::kVc + (mt >> 2) * 512 + (4 * a + b) * 16 + (mt & 3) * 4 + bt] = static_cast<char>(byte);
      }
    }
  } else {
    rec[F::kVc + (4 * (l & 7) + b) * 16 + (l >> 3) * 4 + bt] = static_cast<char>(crumbs);
  }
  if ((l & 7) == 0) {
    const int k = l >> 3;
    *reinterpret_cast<float*>(rec + F::kVm + ((2 * k) * 4 + b) * 16 + 4 * e) = s;
    *reinterpret_cast<float*>(rec + F::kVm + ((2 * k + 1) * 4 + b) * 16 + 4 * e) = lo;
  }
}

__device__ __forceinline__ void copy_row(uint16_t* dst, const uint16_t* src, int part) {
  reinterpret_cast<uint4*>(dst)[part] = reinterpret_cast<const uint4*>(src)[part];
}

// Block-wide exclusive scan of per-sequence work-item counts into pre[0..n].
// Returns false (in every thread) when cu_new / seq_lens_before are malformed:
// cu_new[0] != 0, a decreasing step, cu_new[n] != num_new or a negative length.
// Then no input row is read at all.
__device__ bool build_prefix(const AppendArgs& a, int* pre, int* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  int carry = 0;
  int bad = (a.cu_new[0] != 0 || a.cu_new[a.n] != a.num_new) ? 1 : 0;
  for (int base = 0; base < a.n; base += kThreads) {
    const int i = base + tid;
    int cnt = 0;
    if (i < a.n) {
      const int c0 = a.cu_new[i], c1 = a.cu_new[i + 1];
      const int T0 = a.seq_lens_before[i];
      int ni = c1 - c0;
      if (ni < 0 || T0 < 0 || T0 > (1 << 30) || ni > (1 << 30)) {
        bad = 1;
        ni = 0;
      }
      const int T1 = max(T0, 0) + ni;
      int lo;
      // FP8: one item per (head, 32 new tokens), at least one per head
      cnt = a.bits == 8 ? a.H * max(1, (ni + 31) / 32) : a.H * (1 + tile_range(max(T0, 0), T1, a.R, &lo));
    }
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[w] = x;
    __syncthreads();
    int before = carry;
    for (int q = 0; q < w; ++q) before += warp_tot[q];
    if (i < a.n) pre[i] = before + x - cnt;
    int total = 0;
    for (int q = 0; q < kThreads / 32; ++q) total += warp_tot[q];
    __syncthreads();
    carry += total;
  }
  if (tid == 0) pre[a.n] = carry;
  bad = __syncthreads_or(bad);
  if (bad && blockIdx.x == 0 && tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_CU, a.n);
  return !bad;
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) append_kernel(AppendArgs a) {
  extern __shared__ int pre[];   // [n + 1]
  __shared__ int warp_tot[kThreads / 32];
  __shared__ __align__(16) uint8_t stage[2][1536];
  __shared__ const uint16_t* src[kG];

  if (!build_prefix(a, pre, warp_tot)) return;
  const int total = pre[a.n];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    int lo_i = 0, hi_i = a.n - 1;   // last i with pre[i] <= item
    while (lo_i < hi_i) {
      const int mid = (lo_i + hi_i + 1) >> 1;
      if (pre[mid] <= item) lo_i = mid; else hi_i = mid - 1;
    }
    const int i = lo_i;
    const int T0 = max(a.seq_lens_before[i], 0);
    const int row0 = a.cu_new[i];
    const int ni = max(a.cu_new[i + 1] - row0, 0);
    const int T1 = T0 + ni;
    int tlo;
    const int ntiles = tile_range(T0, T1, a.R, &tlo);
    const int per = 1 + ntiles;
    const int r = item - pre[i];
    const int h = r / per, j = r % per;
    const int slot = a.slot_ids ? a.slot_ids[i] : i;
    if (slot < 0 || slot >= a.max_slots) {
      if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
      continue;
    }
    if (static_cast<long long>(a.bt_stride) * kP < T1) {
      if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, i);
      continue;
    }
    Ctx c{&a, a.block_table + static_cast<long long>(i) * a.bt_stride, slot};
    uint16_t* kring = reinterpret_cast<uint16_t*>(a.kring) + slot * a.kring_slot + h * a.kring_head;
    uint16_t* vring = reinterpret_cast<uint16_t*>(a.vring) + slot * a.vring_slot + h * a.vring_head;
    const int Tk1 = T1 & ~(kG - 1);
    const int Tv0 = max(0, T0 - a.R), Tv1 = max(0, T1 - a.R);

    if (j == 0) {
      // The ring item: every access to this (slot, head)'s rings happens here,
      // reads before writes, so ring rows are never overwritten before use.
      // Its independent reads are issued together first: the stored length, the
      // first value token leaving the window per warp (ring row and page), and
      // each thread's first 16 bytes of the new rows bound for the rings.
      int* len_word = a.lens + slot * a.H + h;
      const int stored = *len_word;
      const int vend = min(T0, Tv1);
      const int tv = Tv0 + warp;
      uint2 vraw = make_uint2(0u, 0u);
      int vpage = 0;
      if (tv < vend) {
        vraw = *reinterpret_cast<const uint2*>(vring + static_cast<long long>(tv % a.R) * kD + 4 * lane);
        vpage = c.bt_row[tv / kP];
      }
      const int kb = max(Tk1, T0), vb = max(T0, Tv1);
      uint4 kfirst = make_uint4(0u, 0u, 0u, 0u), vfirst = kfirst;
      if (tid < (T1 - kb) * 16)
        kfirst = reinterpret_cast<const uint4*>(row_ptr(a.k, row0 + (kb + tid / 16 - T0), a.H, h))[tid % 16];
      if (tid < (T1 - vb) * 16)
        vfirst = reinterpret_cast<const uint4*>(row_ptr(a.v, row0 + (vb + tid / 16 - T0), a.H, h))[tid % 16];
      if (T0 != 0 && stored != T0) {
        if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, i);
        __syncthreads();
        continue;
      }
      const int Tk0 = T0 & ~(kG - 1);
      if (Tk0 < T0 && Tk0 + kG <= T1) {   // first key group mixes ring and new rows
        if (tid < kG) {
          const int t = Tk0 + tid;
          src[tid] = t < T0 ? kring + static_cast<long long>(t % kG) * kD
                            : row_ptr(a.k, row0 + (t - T0), a.H, h);
        }
        __syncthreads();
        key_flush<BITS>(c, h, Tk0 / kG, src, stage);
      }
      if (tv < vend) value_token_row<BITS>(c, h, tv, vraw, vpage);
      for (int t = tv + kThreads / 32; t < vend; t += kThreads / 32)
        value_token<BITS>(c, h, t, vring + static_cast<long long>(t % a.R) * kD);
      __syncthreads();
      for (int q = tid; q < (T1 - kb) * 16; q += kThreads) {
        const int t = kb + q / 16;
        uint16_t* dst = kring + static_cast<long long>(t % kG) * kD;
        if (q == tid) reinterpret_cast<uint4*>(dst)[q % 16] = kfirst;
        else copy_row(dst, row_ptr(a.k, row0 + (t - T0), a.H, h), q % 16);
      }
      for (int q = tid; q < (T1 - vb) * 16; q += kThreads) {
        const int t = vb + q / 16;
        uint16_t* dst = vring + static_cast<long long>(t % a.R) * kD;
        if (q == tid) reinterpret_cast<uint4*>(dst)[q % 16] = vfirst;
        else copy_row(dst, row_ptr(a.v, row0 + (t - T0), a.H, h), q % 16);
      }
      if (tid == 0) *len_word = T1;
      __syncthreads();
    } else {
      const int tile = tlo + j - 1;
      const int t0 = tile * 32;
      if (t0 >= T0 && t0 + kG <= T1) {      // a key group made only of new rows
        if (tid < kG) src[tid] = row_ptr(a.k, row0 + (t0 + tid - T0), a.H, h);
        __syncthreads();
        key_flush<BITS>(c, h, tile, src, stage);
      }
      const int vs = max(t0, T0), ve = min(t0 + 32, Tv1);
      for (int t = vs + warp; t < ve; t += kThreads / 32)
        value_token<BITS>(c, h, t, row_ptr(a.v, row0 + (t - T0), a.H, h));
      __syncthreads();
    }
    (void)lane;
  }
}

// ---- FP8 E4M3 pages ("4.4 KV Cache 量化", sections 4.1 and 4.2) ------------------
// Every new token goes straight to its page: x / scale rounded to fp32, then the
// saturating round-to-nearest-even conversion to E4M3. No ring, no group: an
// item is (sequence, head, 32 new tokens); item 0 of a (sequence, head) checks
// and advances the stored length. Warp w writes tokens w, w + 4, ...; lane l
// owns channels 4l .. 4l+3 of a token (8 bytes of its key row, 8 of its value row).
__device__ __forceinline__ uint32_t e4m3_of(float x, float scale) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fdiv_rn(x, scale), __NV_SATFINITE, __NV_E4M3));
}

__global__ void __launch_bounds__(kThreads) append_fp8_kernel(AppendArgs a) {
  extern __shared__ int pre[];   // [n + 1]
  __shared__ int warp_tot[kThreads / 32];
  if (!build_prefix(a, pre, warp_tot)) return;
  const int total = pre[a.n];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    int lo_i = 0, hi_i = a.n - 1;   // last i with pre[i] <= item
    while (lo_i < hi_i) {
      const int mid = (lo_i + hi_i + 1) >> 1;
      if (pre[mid] <= item) lo_i = mid; else hi_i = mid - 1;
    }
    const int i = lo_i;
    const int T0 = max(a.seq_lens_before[i], 0);
    const int row0 = a.cu_new[i];
    const int ni = max(a.cu_new[i + 1] - row0, 0);
    const int T1 = T0 + ni;
    const int per = max(1, (ni + 31) / 32);
    const int r = item - pre[i];
    const int h = r / per, j = r % per;
    const int slot = a.slot_ids ? a.slot_ids[i] : i;
    if (slot < 0 || slot >= a.max_slots) {
      if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
      continue;
    }
    if (static_cast<long long>(a.bt_stride) * kP < T1) {
      if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, i);
      continue;
    }
    const int* bt_row = a.block_table + static_cast<long long>(i) * a.bt_stride;
    if (j == 0) {
      int* len_word = a.lens + slot * a.H + h;
      const int stored = *len_word;
      if (T0 != 0 && stored != T0) {
        if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, i);
        continue;
      }
      __syncthreads();   // every thread has read the stored length before it changes
      if (tid == 0) *len_word = T1;
    }
    const float ks = a.fp8_scale[h], vs = a.fp8_scale[a.H + h];
    const int n1 = min(ni, 32 * j + 32);
    for (int idx = 32 * j + warp; idx < n1; idx += kThreads / 32) {
      const int t = T0 + idx;
      const int pp = bt_row[t / kP];
      const uint2 kr = *reinterpret_cast<const uint2*>(row_ptr(a.k, row0 + idx, a.H, h) + 4 * lane);
      const uint2 vr = *reinterpret_cast<const uint2*>(row_ptr(a.v, row0 + idx, a.H, h) + 4 * lane);
      if (pp < 0 || pp >= a.num_pages) {
        if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp);
        continue;
      }
      char* rec = a.pages + (static_cast<long long>(pp) * a.H + h) * Rec<8>::kBytes;
      const int tau = t % kP;
      const uint16_t kx[4] = {static_cast<uint16_t>(kr.x & 0xffff), static_cast<uint16_t>(kr.x >> 16),
                              static_cast<uint16_t>(kr.y & 0xffff), static_cast<uint16_t>(kr.y >> 16)};
      const uint16_t vx[4] = {static_cast<uint16_t>(vr.x & 0xffff), static_cast<uint16_t>(vr.x >> 16),
                              static_cast<uint16_t>(vr.y & 0xffff), static_cast<uint16_t>(vr.y >> 16)};
      uint32_t kc[4], vc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        kc[q] = e4m3_of(widen16(kx[q], a.dtype), ks);
        vc[q] = e4m3_of(widen16(vx[q], a.dtype), vs);
      }
      {   // key channels 4l + j: slice kk = l % 8, column b = l / 8; token a + 8 hi
        const int kk = lane & 7, b = lane >> 3;
        const int off = Rec<8>::kKc + (kk >> 1) * 512 + (4 * (tau & 7) + b) * 16 + 8 * (kk & 1) + 2 * (tau >> 3);
        *reinterpret_cast<uint16_t*>(rec + off) = static_cast<uint16_t>(kc[0] | (kc[1] << 8));
        *reinterpret_cast<uint16_t*>(rec + off + 4) = static_cast<uint16_t>(kc[2] | (kc[3] << 8));
      }
      {   // value channel 4l + q = 16 mt + a + 8 up; token tau = 2b + r + 8w
        const int mt = lane >> 2, up = (lane >> 1) & 1;
        const int b = (tau & 7) >> 1, rr = tau & 1, w = tau >> 3;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int aa = 4 * (lane & 1) + q;
          rec[Rec<8>::kVc + (mt >> 1) * 512 + (4 * aa + b) * 16 + 8 * (mt & 1) + 4 * w + 2 * up + rr] =
              static_cast<char>(vc[q]);
        }
      }
    }
  }
}

// Restore of FP8 pages: value(code) * scale, one rounding (as the pages' readers
// see them).
__global__ void __launch_bounds__(kThreads) dequant_fp8_kernel(DequantArgs a) {
  const int h = blockIdx.y;
  const int c = threadIdx.x;
  const int T = a.T;
  if (blockIdx.x == 0 && c == 0 && a.lens[a.slot * a.H + h] != T)
    report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, a.slot);
  const float ks = a.fp8_scale[h], vs = a.fp8_scale[a.H + h];
  for (int t = blockIdx.x * 8; t < min(T, blockIdx.x * 8 + 8); ++t) {
    const int tau = t % kP;
    const int pp = a.bt_row[t / kP];
    const bool ok = pp >= 0 && pp < a.num_pages;
    if (!ok && c == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp);
    float kv = 0.0f, vv = 0.0f;
    if (ok) {
      const char* rec = a.pages + (static_cast<long long>(pp) * a.H + h) * Rec<8>::kBytes;
      const int b = c / 32, kk = (c % 32) / 4, j = c % 4;
      const int koff = Rec<8>::kKc + (kk / 2) * 512 + (4 * (tau % 8) + b) * 16 + 8 * (kk % 2) + 4 * (j / 2) +
                       2 * (tau / 8) + (j % 2);
      const int mt = c / 16, aa = c % 8, up = (c % 16) / 8;
      const int bv = (tau % 8) / 2, rr = tau % 2, w = tau / 8;
      const int voff = Rec<8>::kVc + (mt / 2) * 512 + (4 * aa + bv) * 16 + 8 * (mt % 2) + 4 * w + 2 * up + rr;
      const __half hk = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(rec[koff]), __NV_E4M3);
      const __half hv = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(rec[voff]), __NV_E4M3);
      kv = __fmul_rn(__half2float(hk), ks);
      vv = __fmul_rn(__half2float(hv), vs);
    }
    a.out_k[(static_cast<long long>(h) * T + t) * kD + c] = kv;
    a.out_v[(static_cast<long long>(h) * T + t) * kD + c] = vv;
  }
}

// ---- exact restore -----------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(kThreads) dequant_kernel(DequantArgs a) {
  using F = Rec<BITS>;
  const int h = blockIdx.y;
  const int c = threadIdx.x;
  const int T = a.T;
  const int Tk = T & ~(kG - 1), Tv = max(0, T - a.R);
  if (blockIdx.x == 0 && c == 0 && a.lens[a.slot * a.H + h] != T)
    report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, a.slot);
  const uint16_t* kring = reinterpret_cast<const uint16_t*>(a.kring) + a.slot * a.kring_slot + h * a.kring_head;
  const uint16_t* vring = reinterpret_cast<const uint16_t*>(a.vring) + a.slot * a.vring_slot + h * a.vring_head;
  for (int t = blockIdx.x * 8; t < min(T, blockIdx.x * 8 + 8); ++t) {
    const int tau = t % kP;
    const int pp = a.bt_row[t / kP];
    const bool ok = pp >= 0 && pp < a.num_pages;
    if (!ok && c == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp);
    const char* rec = ok ? a.pages + (static_cast<long long>(pp) * a.H + h) * F::kBytes : nullptr;
    float kv = 0.0f, vv = 0.0f;
    if (t < Tk) {
      const int grp = t / kG;
      const int pp2 = a.bt_row[2 * grp + c / 64];
      const bool ok2 = pp2 >= 0 && pp2 < a.num_pages;
      if (ok && ok2) {
        const char* rec2 = a.pages + (static_cast<long long>(pp2) * a.H + h) * F::kBytes;
        const int L = 4 * (tau & 7) + c / 32, kk = (c % 32) / 4, j = c % 4;
        const int bj = (j == 0) ? 0 : (j == 1) ? 2 : (j == 2) ? 1 : 3;
        int code;
        if constexpr (BITS == 4) {
          const uint8_t byte = static_cast<uint8_t>(rec[F::kKc + (kk / 4) * 512 + L * 16 + (kk % 4) * 4 + bj]);
          code = tau >= 8 ? (byte >> 4) : (byte & 15);
        } else {
          const uint8_t byte = static_cast<uint8_t>(rec[F::kKc + L * 16 + (kk / 2) * 4 + bj]);
          code = (byte >> (2 * (2 * (kk & 1) + (tau >= 8 ? 1 : 0)))) & 3;
        }
        const int cl = c % 64, u = cl / 32, i = (cl % 32) / 4, e = cl % 4;
        const float s = *reinterpret_cast<const float*>(rec2 + F::kKm + (2 * i + u) * 16 + 4 * e);
        const float mn = *reinterpret_cast<const float*>(rec2 + F::kKm + (2 * i + u) * 16 + 4 * e + 256);
        kv = __fmaf_rn(static_cast<float>(code), s, mn);
      }
    } else {
      kv = widen16(kring[static_cast<long long>(t % kG) * kD + c], a.dtype);
    }
    if (t < Tv) {
      if (ok) {
        const int mt = c / 16, aa = c % 8, high = (c % 16) / 8;
        const int b = (tau & 7) >> 1, wv = tau >> 3, r = tau & 1;
        const int bt = wv ? (r ? 3 : 1) : (r ? 2 : 0);
        int code;
        if constexpr (BITS == 4) {
          const uint8_t byte = static_cast<uint8_t>(
              rec[F::kVc + (mt / 4) * 512 + (4 * aa + b) * 16 + (mt % 4) * 4 + bt]);
          code = high ? (byte >> 4) : (byte & 15);
        } else {
          const uint8_t byte = static_cast<uint8_t>(rec[F::kVc + (4 * aa + b) * 16 + (c / 32) * 4 + bt]);
          code = (byte >> (2 * ((c % 32) / 8))) & 3;
        }
        const int k = c / 32, e = r + 2 * wv;
        const float s = *reinterpret_cast<const float*>(rec + F::kVm + ((2 * k) * 4 + b) * 16 + 4 * e);
        const float mn = *reinterpret_cast<const float*>(rec + F::kVm + ((2 * k + 1) * 4 + b) * 16 + 4 * e);
        vv = __fmaf_rn(static_cast<float>(code), s, mn);
      }
    } else {
      vv = widen16(vring[static_cast<long long>(t % a.R) * kD + c], a.dtype);
    }
    a.out_k[(static_cast<long long>(h) * T + t) * kD + c] = kv;
    a.out_v[(static_cast<long long>(h) * T + t) * kD + c] = vv;
  }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, int grid, cudaStream_t st) {
  if (a.n <= 0 || grid <= 0) return cudaSuccess;
  if (a.n > kMaxSeqsPerCall) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(a.n + 1) * sizeof(int);
  if (a.bits == 8) append_fp8_kernel<<<grid, kThreads, smem, st>>>(a);
  else if (a.bits == 2) append_kernel<2><<<grid, kThreads, smem, st>>>(a);
  else append_kernel<4><<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const DequantArgs& a, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  dim3 grid((a.T + 7) / 8, a.H);
  if (a.bits == 8) dequant_fp8_kernel<<<grid, kThreads, 0, st>>>(a);
  else if (a.bits == 2) dequant_kernel<2><<<grid, kThreads, 0, st>>>(a);
  else dequant_kernel<4><<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace s4kv
