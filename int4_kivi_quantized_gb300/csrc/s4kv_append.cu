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
#include "s4kv_quant.cuh"

#include <cuda_fp8.h>
#include <climits>
#include <mutex>

namespace s4kv {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxSeqsPerCall = 8192;
constexpr int kMaxAppendDevices = 64;

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
      const int lo_c = quant::code<BITS>(x[16 * p + a], lo, s);
      const int hi_c = quant::code<BITS>(x[16 * p + a + 8], lo, s);
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
// already loaded (the shared warp routine of s4kv_quant.cuh).
template <int BITS>
__device__ void value_token_row(const Ctx& c, int h, int t, uint2 raw, int pp) {
  char* rec = nullptr;
  if (pp < 0 || pp >= c.a->num_pages) {
    if ((threadIdx.x & 31) == 0) report(c.a->status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp);
  } else {
    rec = c.a->pages + (static_cast<long long>(pp) * c.a->H + h) * Rec<BITS>::kBytes;
  }
  quant::value_token<BITS>(rec, t, raw, c.a->dtype);
}

// Block-wide exclusive scan of per-sequence work-item counts into pre[0..n].
// Returns false (in every thread) when cu_new / seq_lens_before are malformed:
// cu_new[0] != 0, a decreasing step, cu_new[n] != num_new or a negative length.
// Then no input row is read at all.
// With seq (tile kernel), also keeps each sequence's length before the append
// (seq[i]) and first new row (seq[n + 1 + i], and seq[2n + 1] = cu_new[n]) in
// shared memory, so that work items are decoded without global loads.
// Work weight of a ring item in tile units: one, plus one per kRingTokensPerUnit
// value tokens it quantizes as they leave the window (token by token, the
// slowest work of a chunk append).
constexpr int kRingTokensPerUnit = 16;
__device__ __forceinline__ int ring_weight(int T0, int T1, int R) {
  const int Tv0 = max(0, T0 - R), Tv1 = max(0, T1 - R);
  const int leaving = max(0, min(T0, Tv1) - Tv0);
  return 1 + (leaving + kRingTokensPerUnit - 1) / kRingTokensPerUnit;
}

// Per-sequence prefixes of the call's items (pre) and, for KIVI pages, of their
// work (cpre: a ring item weighs ring_weight, a tile one). Sequence i owns
// H (1 + tiles) items, head-major, each head's ring item first.
__device__ bool build_prefix(const AppendArgs& a, int* pre, int* warp_tot, int* seq = nullptr,
                             int* cpre = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  __shared__ int warp_cost[kThreads / 32];
  int carry = 0, ccarry = 0;
  int bad = (a.cu_new[0] != 0 || a.cu_new[a.n] != a.num_new) ? 1 : 0;
  for (int base = 0; base < a.n; base += kThreads) {
    const int i = base + tid;
    int cnt = 0, cost = 0;
    if (i < a.n) {
      const int c0 = a.cu_new[i], c1 = a.cu_new[i + 1];
      const int T0 = a.seq_lens_before[i];
      if (seq) {
        seq[i] = max(T0, 0);
        seq[a.n + 1 + i] = c0;
        if (i == a.n - 1) seq[2 * a.n + 1] = c1;
      }
      int ni = c1 - c0;
      if (ni < 0 || T0 < 0 || T0 > (1 << 30) || ni > (1 << 30)) {
        bad = 1;
        ni = 0;
      }
      const int T1 = max(T0, 0) + ni;
      int lo;
      // FP8: one item per (head, 32 new tokens), at least one per head
      if (a.bits == 8) {
        cnt = a.H * max(1, (ni + 31) / 32);
      } else {
        const int tiles = tile_range(max(T0, 0), T1, a.R, &lo);
        cnt = a.H * (1 + tiles);
        cost = a.H * (ring_weight(max(T0, 0), T1, a.R) + tiles);
      }
    }
    int x = cnt, y = cost;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, x, o);
      const int v = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) {
        x += u;
        y += v;
      }
    }
    if (lane == 31) {
      warp_tot[w] = x;
      warp_cost[w] = y;
    }
    __syncthreads();
    int before = carry, cbefore = ccarry;
    for (int q = 0; q < w; ++q) {
      before += warp_tot[q];
      cbefore += warp_cost[q];
    }
    if (i < a.n) {
      pre[i] = before + x - cnt;
      if (cpre) cpre[i] = cbefore + y - cost;
    }
    int total = 0, ctotal = 0;
    for (int q = 0; q < kThreads / 32; ++q) {
      total += warp_tot[q];
      ctotal += warp_cost[q];
    }
    __syncthreads();
    carry += total;
    ccarry += ctotal;
  }
  if (tid == 0) {
    pre[a.n] = carry;
    if (cpre) cpre[a.n] = ccarry;
  }
  bad = __syncthreads_or(bad);
  if (bad && blockIdx.x == 0 && tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_CU, a.n);
  return !bad;
}

// ---- whole 32-token tiles of new rows (chunk appends) ---------------------------
// A tile item whose key group is made only of new rows takes this path. Its key
// and value rows arrive by cp.async in a two-stage ring (the CTA's next tile
// loads while this one is quantized). Warps 0-1 quantize the keys, warps 2-3 the
// values, each pair assembling its half of the tile's two page records in shared
// memory and writing it with 16-byte stores. The tile owns both pages (its 32
// tokens are all new), so whole records are written. Value bytes of tokens that
// are still inside the residual window are written as well, from the same rows:
// those bytes are undefined until the token leaves the window, and then they are
// rewritten with the same values.
//
// The code of x is rne(fl(fl(x - min) / s)). Per element this path computes
// t' = fl(fl(x - min) * r) with r = fl(1 / s) (correctly rounded), two
// elements per instruction (packed fp32 pairs). The difference fl(x - min) is
// the division's own numerator, so against the quotient q = fl(x - min) / s:
//   |t' - q| <= 2^-24 |t'| + |fl(x - min)| |r - 1/s| <= 2^-20 + 2^-20 = 2^-19
// for quotients below 16, and fl(q) is within 2^-21 of q. So whenever t' is
// farther than 2^-17 from every half-integer, t' and fl(q) lie strictly between
// the same two half-integers and round to the same integer (4-bit codes: 0..15;
// 2-bit: 0..3). Elements that fail this test, and groups whose s is so small
// that 1 / s is not used (below 2^-100), are recomputed with the IEEE division
// itself, so the codes are exactly those of the division.

constexpr int kTileRowBytes = kD * 2;                  // one 16-bit row
constexpr int kTileBytes = kG * kTileRowBytes;         // 32 rows: 8 KiB
constexpr int kStageBytes = 2 * kTileBytes;            // key tile, value tile
#ifndef S4KV_APPEND_STAGES
#define S4KV_APPEND_STAGES 2
#endif
#ifndef S4KV_APPEND_CTAS
#define S4KV_APPEND_CTAS 3
#endif
constexpr int kNumStages = S4KV_APPEND_STAGES;   // tiles a CTA holds: one being quantized, the rest loading
constexpr int kAppendCtas = S4KV_APPEND_CTAS;    // resident CTAs per SM the launch is sized for
static_assert(kNumStages == 2 || kNumStages == 3, "one or two tiles in flight");
constexpr int kRecPad = 64;                            // the second staged record starts 16 banks on
constexpr int kStagingBytes = 2 * Rec<4>::kBytes + kRecPad + 64;
constexpr int kParamFloats = 4 * kD;                   // key lo, s, 1/s, -lo/s per channel

// Dynamic shared memory: [prefix (n + 1) ints, 128-byte padded][stages][staging][key params].
// prefix [n + 1], then the per-sequence copies of build_prefix (2n + 2 ints)
// and the work prefix cpre [n + 1]
__host__ __device__ constexpr int prefix_bytes(int n) {
  return 2 * (((n + 1) * 4 + 127) & ~127) + (((2 * n + 2) * 4 + 127) & ~127);
}
__host__ __device__ constexpr int seq_info_offset(int n) { return ((n + 1) * 4 + 127) & ~127; }
__host__ __device__ constexpr int cost_prefix_offset(int n) {
  return seq_info_offset(n) + (((2 * n + 2) * 4 + 127) & ~127);
}
__host__ __device__ constexpr int append_smem_bytes(int n) {
  return prefix_bytes(n) + kNumStages * kStageBytes + kStagingBytes + kParamFloats * 4;
}

constexpr float kRoundMagic = 12582912.0f;             // 1.5 * 2^23: t + this rounds t to an integer (half even)
constexpr float kTieGuard = 0.4999923706054688f;       // 0.5 - 2^-17

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// waits for all but the newest kNumStages - 1 groups of this thread
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group %0;" ::"n"(kNumStages - 1) : "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Byte offset of 16-byte chunk q (0..15) of row t in a staged tile. The chunk
// index is XORed with t % 8, so the eight rows that one quarter of a warp reads
// at the same chunk fall in different banks, and with 4 for rows 16..31, so that
// rows t and t + 16 (read together by the two halves of a warp) do too.
__device__ __forceinline__ int sw_off(int t, int q) {
  return t * kTileRowBytes + ((q ^ (t & 7) ^ ((t >> 2) & 4)) << 4);
}

template <int DT>
__device__ __forceinline__ float lo_of(uint32_t w) {
  if constexpr (DT == S4KV_BF16) return __uint_as_float(w << 16);
  else return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}
template <int DT>
__device__ __forceinline__ float hi_of(uint32_t w) {
  if constexpr (DT == S4KV_BF16) return __uint_as_float(w & 0xffff0000u);
  else return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}
template <int DT>
__device__ __forceinline__ float elem(const uint32_t* x, int c) {   // element c of packed pairs
  return (c & 1) ? hi_of<DT>(x[c >> 1]) : lo_of<DT>(x[c >> 1]);
}
// Elementwise min / max of two packed 16-bit pairs (exact, like the fp32 compare
// of the widened values; a signed zero may come out either way and is
// canonicalised afterwards).
template <int DT>
__device__ __forceinline__ uint32_t min2(uint32_t x, uint32_t y) {
  if constexpr (DT == S4KV_BF16) {
    const __nv_bfloat162 r = __hmin2(*reinterpret_cast<const __nv_bfloat162*>(&x),
                                     *reinterpret_cast<const __nv_bfloat162*>(&y));
    return *reinterpret_cast<const uint32_t*>(&r);
  } else {
    const __half2 r = __hmin2(*reinterpret_cast<const __half2*>(&x), *reinterpret_cast<const __half2*>(&y));
    return *reinterpret_cast<const uint32_t*>(&r);
  }
}
template <int DT>
__device__ __forceinline__ uint32_t max2(uint32_t x, uint32_t y) {
  if constexpr (DT == S4KV_BF16) {
    const __nv_bfloat162 r = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&x),
                                     *reinterpret_cast<const __nv_bfloat162*>(&y));
    return *reinterpret_cast<const uint32_t*>(&r);
  } else {
    const __half2 r = __hmax2(*reinterpret_cast<const __half2*>(&x), *reinterpret_cast<const __half2*>(&y));
    return *reinterpret_cast<const uint32_t*>(&r);
  }
}

// Four byte values (low bytes of b0..b3) into one word, in the record's byte
// order for channels c0, c1, c2, c3: byte 0 <- c0, 1 <- c2, 2 <- c1, 3 <- c3.
__device__ __forceinline__ uint32_t word_0213(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b2, 0x0040), __byte_perm(b1, b3, 0x0040), 0x5410);
}

// 1 / s for the per-element path (0 when s == 0: every code 0); slow is set
// when the group must take the division instead (s below 2^-100).
__device__ __forceinline__ float recip_param(float s, bool& slow) {
  slow = s != 0.0f && s < 7.8886091e-31f;
  return (s == 0.0f || slow) ? 0.0f : __frcp_rn(s);
}

// Codes of two elements (x.x, x.y) with the group minima (mlo = -min) and
// reciprocal scales r per element, in the low bits of the two returned words;
// worst collects the largest distance |t' - rne(t')| seen.
__device__ __forceinline__ uint2 code_pair(float2 x, float2 mlo, float2 r, float& worst) {
  const float2 kM = make_float2(kRoundMagic, kRoundMagic);
  const float2 kNegM = make_float2(-kRoundMagic, -kRoundMagic);
  const float2 kNeg1 = make_float2(-1.0f, -1.0f);
  const float2 t = __fmul2_rn(__fadd2_rn(x, mlo), r);
  const float2 y = __fadd2_rn(t, kM);
  const float2 f = __fadd2_rn(y, kNegM);           // rne(t), exact
  const float2 d = __ffma2_rn(t, kNeg1, f);        // f - t, exact
  worst = fmaxf(worst, fmaxf(fabsf(d.x), fabsf(d.y)));
  return make_uint2(__float_as_uint(y.x), __float_as_uint(y.y));
}

template <int DT>
__device__ __forceinline__ float2 widen2(uint32_t w) { return make_float2(lo_of<DT>(w), hi_of<DT>(w)); }

template <int DT>
__device__ __forceinline__ float elem16(const uint8_t* tile, int t, int c) {   // element c of row t
  const uint16_t v = reinterpret_cast<const uint16_t*>(tile + sw_off(t, c >> 3))[c & 7];
  return DT == S4KV_BF16 ? __uint_as_float(static_cast<uint32_t>(v) << 16) : __half2float(__ushort_as_half(v));
}

// Key code words whose flag is set (bit m: word m of the lane's 16 channels
// c0 .. c0+15, rows ra and ra + 8), recomputed with the IEEE division and
// written over the per-element results at dst. 4-bit: word m holds channels
// c0 + 4m .. c0 + 4m + 3 (dst: one 16-byte chunk); 2-bit: word h holds
// channels c0 + 8h + 0..3 and + 4..7 (dst: two words). lo, s: the channels'
// parameters, indexed from c0.
template <int BITS, int DT>
__device__ __noinline__ void key_words_fix(unsigned flags, const uint8_t* Ks, int ra, int c0, const float* lo,
                                           const float* s, uint8_t* dst) {
  constexpr int kPer = BITS == 4 ? 4 : 8;   // channels per word
  while (flags) {
    const int m = __ffs(flags) - 1;
    flags &= flags - 1;
    uint32_t B[4];
    for (int j = 0; j < 4; ++j) {
      if constexpr (BITS == 4) {
        const int c = kPer * m + j;
        B[j] = quant::code<4>(elem16<DT>(Ks, ra, c0 + c), lo[c], s[c]) |
               (quant::code<4>(elem16<DT>(Ks, ra + 8, c0 + c), lo[c], s[c]) << 4);
      } else {
        const int c = kPer * m + j, c4 = c + 4;
        B[j] = quant::code<2>(elem16<DT>(Ks, ra, c0 + c), lo[c], s[c]) |
               (quant::code<2>(elem16<DT>(Ks, ra + 8, c0 + c), lo[c], s[c]) << 2) |
               (quant::code<2>(elem16<DT>(Ks, ra, c0 + c4), lo[c4], s[c4]) << 4) |
               (quant::code<2>(elem16<DT>(Ks, ra + 8, c0 + c4), lo[c4], s[c4]) << 6);
      }
    }
    reinterpret_cast<uint32_t*>(dst)[m] = word_0213(B[0], B[1], B[2], B[3]);
  }
}

// Value code bytes a = 2i, 2i + 1 of token t, group k (channels 32k .. 32k+31)
// for every flagged i, recomputed with the IEEE division and written over the
// per-element results at vc (the token's byte of the group's first word; the
// byte of column a is a * 64 further, the second 4-bit word 4 further).
template <int BITS, int DT>
__device__ __noinline__ void value_bytes_fix(unsigned flags, const uint8_t* Vs, int t, int k, float lo, float s,
                                             uint8_t* vc) {
  while (flags) {
    const int i = __ffs(flags) - 1;
    flags &= flags - 1;
    for (int aa = 2 * i; aa < 2 * i + 2; ++aa) {
      if constexpr (BITS == 4) {
        for (int x = 0; x < 2; ++x) {
          const int c = 32 * k + 16 * x + aa;
          vc[4 * x + aa * 64] = static_cast<uint8_t>(quant::code<4>(elem16<DT>(Vs, t, c), lo, s) |
                                                     (quant::code<4>(elem16<DT>(Vs, t, c + 8), lo, s) << 4));
        }
      } else {
        uint32_t v = 0;
        for (int q = 0; q < 4; ++q) v |= quant::code<2>(elem16<DT>(Vs, t, 32 * k + 8 * q + aa), lo, s) << (2 * q);
        vc[aa * 64] = static_cast<uint8_t>(v);
      }
    }
  }
}

struct Item {
  int i, h, j, T0, T1, row0, tile;   // tile: index of the 32-token tile (items j >= 1)
  bool fast;                         // a tile whose key group is made only of new rows
};

__device__ __forceinline__ Item item_of(const AppendArgs& a, const int* pre, const int* seq, int item) {
  Item it;
  int lo_i = 0, hi_i = a.n - 1;   // last i with pre[i] <= item
  while (lo_i < hi_i) {
    const int mid = (lo_i + hi_i + 1) >> 1;
    if (pre[mid] <= item) lo_i = mid; else hi_i = mid - 1;
  }
  it.i = lo_i;
  it.T0 = seq[it.i];
  it.row0 = seq[a.n + 1 + it.i];
  it.T1 = it.T0 + max(seq[a.n + 2 + it.i] - it.row0, 0);
  int tlo;
  const int per = 1 + tile_range(it.T0, it.T1, a.R, &tlo);
  const int r = item - pre[it.i];
  // r / per through a float quotient (off by at most one, then corrected)
  int h = __float2int_rz(__fdividef(static_cast<float>(r), static_cast<float>(per)));
  if (h * per > r) --h;
  else if ((h + 1) * per <= r) ++h;
  it.h = h;
  it.j = r - h * per;
  it.tile = tlo + it.j - 1;
  it.fast = it.j >= 1 && kG * it.tile >= it.T0 && kG * it.tile + kG <= it.T1;
  return it;
}

// First item whose share of the work line starts at or after x: the work line
// lays the items end to end in item order, a ring item weighing ring_weight and
// a tile one (cpre: per-sequence prefix). A CTA takes the items that start in its
// slice of the line, so CTAs that draw ring items with many leaving value tokens
// take fewer tiles.
__device__ __forceinline__ int item_from_cost(const AppendArgs& a, const int* pre, const int* seq, const int* cpre,
                                              long long x) {
  if (x >= cpre[a.n]) return pre[a.n];
  int lo = 0, hi = a.n - 1;   // last sequence with cpre <= x (every sequence weighs at least H)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cpre[mid] <= x) lo = mid; else hi = mid - 1;
  }
  const int T0 = seq[lo], T1 = T0 + max(seq[a.n + 2 + lo] - seq[a.n + 1 + lo], 0);
  const int per = (pre[lo + 1] - pre[lo]) / a.H;   // 1 + tiles
  const int wr = ring_weight(T0, T1, a.R);
  const int unit = wr + per - 1;                    // one head's work
  const int off = static_cast<int>(x - cpre[lo]);
  const int h = off / unit, within = off - h * unit;
  // the ring item starts at 0, tile j >= 1 at wr + j - 1
  int j = within == 0 ? 0 : max(1, within - wr + 1);
  if (j >= per) return pre[lo] + (h + 1) * per;   // the next head's ring item (or the next sequence)
  return pre[lo] + h * per + j;
}

// Issues the cp.async copies of a fast tile's key and value rows into a stage.
// The rows of a whole new tile into its stage, and (thread 0) the tile's slot
// and its two pool pages into ref[0..2], all in the calling threads' current
// cp.async group. A table too narrow for the tile leaves ref alone (the tile
// reports it and writes nothing).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void tile_prefetch(const AppendArgs& a, const Item& it, uint8_t* stage, int* ref) {
  if (threadIdx.x == 0 && static_cast<long long>(a.bt_stride) * kP >= it.T1) {
    const int* bt_row = a.block_table + static_cast<long long>(it.i) * a.bt_stride;
    if (a.slot_ids) cp_async4(ref, a.slot_ids + it.i);
    else ref[0] = it.i;
    cp_async4(ref + 1, bt_row + 2 * it.tile);
    cp_async4(ref + 2, bt_row + 2 * it.tile + 1);
  }
  // thread: chunk q of rows t, t + 8, t + 16, t + 24
  const int t = threadIdx.x >> 4, q = threadIdx.x & 15;
  const long long row = it.row0 + (kG * it.tile - it.T0) + t;
  const long long off = (row * a.H + it.h) * kD + q * 8;
  const long long step = 8LL * a.H * kD;   // 8 rows
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    uint8_t* dst = stage + sw_off(t + 8 * x, q);
    cp_async16(dst, a.k + off + x * step);
    cp_async16(dst + kTileBytes, a.v + off + x * step);
  }
}

// One lane's value group: channels 32k .. 32k+31 of the row `row` of a staged
// 32-row tile (`Vs`, the swizzled layout of tile_prefetch), which holds token
// `tok`; its scale, min and codes go into `rec`, the record of the token's page
// (staged or in the pool): min/max over the lane's 32 values, the reciprocal path
// with the division where an element is next to a half-integer.
template <int BITS, int DT>
__device__ __noinline__ void value_lane(const uint8_t* Vs, int row, int tok, uint8_t* rec, int k) {
  using F = Rec<BITS>;
  const int tau = tok & 15;
  const int b = (tau & 7) >> 1, e = (tau & 1) + 2 * (tau >> 3);
  const int pos = (tau & 1) * 2 + (tau >> 3);   // byte of this token in a value word
  uint32_t xv[16];
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(xv + 4 * q) = *reinterpret_cast<const uint4*>(Vs + sw_off(row, 4 * k + q));
  uint32_t mn = xv[0], mx = xv[0];
#pragma unroll
  for (int x = 1; x < 16; ++x) {
    mn = min2<DT>(mn, xv[x]);
    mx = max2<DT>(mx, xv[x]);
  }
  const float lo = __fadd_rn(fminf(lo_of<DT>(mn), hi_of<DT>(mn)), 0.0f);
  const float hi = __fadd_rn(fmaxf(lo_of<DT>(mx), hi_of<DT>(mx)), 0.0f);
  const float sc = __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(F::kLevels));
  bool vslow;
  const float rcp = recip_param(sc, vslow);
  float* vm = reinterpret_cast<float*>(rec + F::kVm);
  vm[(((2 * k) * 4 + b) * 16 + 4 * e) / 4] = sc;
  vm[(((2 * k + 1) * 4 + b) * 16 + 4 * e) / 4] = lo;
  const float2 r2 = make_float2(rcp, rcp), n2 = make_float2(-lo, -lo);
  uint8_t* vc = rec + F::kVc + b * 16 + pos + (BITS == 4 ? (k >> 1) * 512 + (2 * k & 3) * 4 : k * 4);
  unsigned flags = 0;   // byte pairs with an element next to a half-integer
#pragma unroll
  for (int i = 0; i < 4; ++i) {   // bytes a = 2i, 2i + 1
    float worst = 0.0f;
    if constexpr (BITS == 4) {
#pragma unroll
      for (int x = 0; x < 2; ++x) {   // word of channels 32k + 16x + a (low) and + 8 (high)
        const uint2 lo2 = code_pair(widen2<DT>(xv[8 * x + i]), n2, r2, worst);
        const uint2 hi2 = code_pair(widen2<DT>(xv[8 * x + 4 + i]), n2, r2, worst);
        vc[4 * x + 2 * i * 64] = static_cast<uint8_t>(lo2.x + (hi2.x << 4));
        vc[4 * x + (2 * i + 1) * 64] = static_cast<uint8_t>(lo2.y + (hi2.y << 4));
      }
    } else {
      uint2 q[4];   // channels 32k + 8qq + 2i, + 1
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) q[qq] = code_pair(widen2<DT>(xv[4 * qq + i]), n2, r2, worst);
      vc[2 * i * 64] = static_cast<uint8_t>(q[0].x + (q[1].x << 2) + (q[2].x << 4) + (q[3].x << 6));
      vc[(2 * i + 1) * 64] = static_cast<uint8_t>(q[0].y + (q[1].y << 2) + (q[2].y << 4) + (q[3].y << 6));
    }
    flags |= (worst > kTieGuard ? 1u : 0u) << i;
  }
  if (vslow) flags = 0xfu;
  if (flags) value_bytes_fix<BITS, DT>(flags, Vs, row, k, lo, sc, vc);
}

template <int BITS, int DT>
__device__ void fast_tile(const AppendArgs& a, const Item& it, const uint8_t* stage, const int* tile_ref,
                          uint8_t* staging, float* prm) {
  using F = Rec<BITS>;
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  if (static_cast<long long>(a.bt_stride) * kP < it.T1) {
    if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, it.i);
    return;
  }
  // tile_ref: the slot and the tile's two pool pages, loaded with the tile's rows
  // (tile_prefetch) and checked before the records are written
  uint8_t* const st0 = staging;
  uint8_t* const st1 = staging + F::kBytes + kRecPad;
  const uint8_t* Ks = stage;
  const uint8_t* Vs = stage + kTileBytes;
  float* klo = prm;
  float* ks = prm + kD;
  float* kr = prm + 2 * kD;
  float* kn = prm + 3 * kD;   // -min
  bool kslow;                 // some channel of this warp takes the division

  // ---- keys, channels 32w .. 32w+31: per-channel groups over the 32 tokens --
  {
    const int cp = 16 * w + (l & 15), half = l >> 4;   // channel pair, rows 16 half .. 16 half + 15
    // row 16 half + i sits at this base plus i * 256 (i and i + 8 share the swizzle)
    const uint8_t* kb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) kb[i] = Ks + sw_off(16 * half + i, cp >> 2) + (cp & 3) * 4;
    uint32_t mn = *reinterpret_cast<const uint32_t*>(kb[0]), mx = mn;
#pragma unroll
    for (int i = 1; i < 16; ++i) {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(kb[i & 7] + (i >> 3) * 8 * kTileRowBytes);
      mn = min2<DT>(mn, v);
      mx = max2<DT>(mx, v);
    }
    mn = min2<DT>(mn, __shfl_xor_sync(0xffffffffu, mn, 16));
    mx = max2<DT>(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const int ch = 2 * cp + half;   // this lane's channel
    const float lo = __fadd_rn(half ? hi_of<DT>(mn) : lo_of<DT>(mn), 0.0f);
    const float hi = __fadd_rn(half ? hi_of<DT>(mx) : lo_of<DT>(mx), 0.0f);
    const float sc = __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(F::kLevels));
    bool slow;
    const float rcp = recip_param(sc, slow);
    kslow = __any_sync(0xffffffffu, slow);
    klo[ch] = lo;
    ks[ch] = sc;
    kr[ch] = rcp;
    kn[ch] = -lo;
    const int u = (ch >> 5) & 1, i = (ch >> 2) & 7, ee = ch & 3;
    float* meta = reinterpret_cast<float*>(((ch >> 6) ? st1 : st0) + F::kKm);
    meta[((2 * i + u) * 16 + 4 * ee) / 4] = sc;
    meta[((2 * i + u) * 16 + 4 * ee + 256) / 4] = lo;
  }
  __syncwarp();
  {
    // 16 channels c0 .. c0+15 of rows ra (low codes) and ra + 8 (high codes);
    // the per-element results are stored at once and overwritten by the
    // division's when some element needs it
    const int aa = l & 7, hh = (l >> 3) & 1, p = l >> 4;
    const int c0 = 32 * w + 16 * hh, ra = 16 * p + aa;
    uint32_t xa[8], xb[8];
    *reinterpret_cast<uint4*>(xa) = *reinterpret_cast<const uint4*>(Ks + sw_off(ra, c0 >> 3));
    *reinterpret_cast<uint4*>(xa + 4) = *reinterpret_cast<const uint4*>(Ks + sw_off(ra, (c0 >> 3) + 1));
    *reinterpret_cast<uint4*>(xb) = *reinterpret_cast<const uint4*>(Ks + sw_off(ra + 8, c0 >> 3));
    *reinterpret_cast<uint4*>(xb + 4) = *reinterpret_cast<const uint4*>(Ks + sw_off(ra + 8, (c0 >> 3) + 1));
    // codes of channel pair i: token ra, token ra + 8
    auto pair_codes = [&](int i, uint2& qa, uint2& qb, float& worst) {
      const float2 r2 = *reinterpret_cast<const float2*>(kr + c0 + 2 * i);
      const float2 n2 = *reinterpret_cast<const float2*>(kn + c0 + 2 * i);
      qa = code_pair(widen2<DT>(xa[i]), n2, r2, worst);
      qb = code_pair(widen2<DT>(xb[i]), n2, r2, worst);
    };
    uint8_t* stp = p ? st1 : st0;
    unsigned flags = 0;   // words with an element next to a half-integer
    if constexpr (BITS == 4) {
      uint32_t wd[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {   // channels c0 + 4m .. c0 + 4m + 3
        uint2 a0, b0, a1, b1;
        float worst = 0.0f;
        pair_codes(2 * m, a0, b0, worst);
        pair_codes(2 * m + 1, a1, b1, worst);
        wd[m] = word_0213(a0.x + (b0.x << 4), a0.y + (b0.y << 4), a1.x + (b1.x << 4), a1.y + (b1.y << 4));
        flags |= (worst > kTieGuard ? 1u : 0u) << m;
      }
      uint8_t* dst = stp + F::kKc + hh * 512 + (4 * aa + w) * 16;
      *reinterpret_cast<uint4*>(dst) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      if (kslow) flags = 0xfu;
      if (flags) key_words_fix<4, DT>(flags, Ks, ra, c0, klo + c0, ks + c0, dst);
    } else {
      uint32_t wd[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {   // channels c0 + 8 h2 + j (slice 2kp) and + 4 + j (slice 2kp + 1)
        uint2 qa[4], qb[4];
        float worst = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) pair_codes(4 * h2 + i, qa[i], qb[i], worst);
        uint32_t B[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t a_lo = (j & 1) ? qa[j >> 1].y : qa[j >> 1].x;
          const uint32_t b_lo = (j & 1) ? qb[j >> 1].y : qb[j >> 1].x;
          const uint32_t a_hi = (j & 1) ? qa[2 + (j >> 1)].y : qa[2 + (j >> 1)].x;
          const uint32_t b_hi = (j & 1) ? qb[2 + (j >> 1)].y : qb[2 + (j >> 1)].x;
          B[j] = a_lo + (b_lo << 2) + (a_hi << 4) + (b_hi << 6);
        }
        wd[h2] = word_0213(B[0], B[1], B[2], B[3]);
        flags |= (worst > kTieGuard ? 1u : 0u) << h2;
      }
      uint8_t* dst = stp + F::kKc + (4 * aa + w) * 16 + 8 * hh;
      *reinterpret_cast<uint2*>(dst) = make_uint2(wd[0], wd[1]);
      if (kslow) flags = 0x3u;
      if (flags) key_words_fix<2, DT>(flags, Ks, ra, c0, klo + c0, ks + c0, dst);
    }
  }

  // ---- values, token t = 8w + l % 8, group k = l / 8 (channels 32k .. 32k+31) --
  // (value_lane's computation, inline: the tile's key and value work then share
  // one instruction schedule)
  {
    const int t = 8 * w + (l & 7), k = l >> 3;
    const int tau = t & 15;
    const int b = (tau & 7) >> 1, e = (tau & 1) + 2 * (tau >> 3);
    const int pos = (tau & 1) * 2 + (tau >> 3);   // byte of this token in a value word
    uint8_t* stp = (t >> 4) ? st1 : st0;
    uint32_t xv[16];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(xv + 4 * q) = *reinterpret_cast<const uint4*>(Vs + sw_off(t, 4 * k + q));
    uint32_t mn = xv[0], mx = xv[0];
#pragma unroll
    for (int x = 1; x < 16; ++x) {
      mn = min2<DT>(mn, xv[x]);
      mx = max2<DT>(mx, xv[x]);
    }
    const float lo = __fadd_rn(fminf(lo_of<DT>(mn), hi_of<DT>(mn)), 0.0f);
    const float hi = __fadd_rn(fmaxf(lo_of<DT>(mx), hi_of<DT>(mx)), 0.0f);
    const float sc = __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(F::kLevels));
    bool vslow;
    const float rcp = recip_param(sc, vslow);
    float* vm = reinterpret_cast<float*>(stp + F::kVm);
    vm[(((2 * k) * 4 + b) * 16 + 4 * e) / 4] = sc;
    vm[(((2 * k + 1) * 4 + b) * 16 + 4 * e) / 4] = lo;
    const float2 r2 = make_float2(rcp, rcp), n2 = make_float2(-lo, -lo);
    uint8_t* vc = stp + F::kVc + b * 16 + pos +
                  (BITS == 4 ? (k >> 1) * 512 + (2 * k & 3) * 4 : k * 4);
    unsigned flags = 0;   // byte pairs with an element next to a half-integer
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // bytes a = 2i, 2i + 1
      float worst = 0.0f;
      if constexpr (BITS == 4) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {   // word of channels 32k + 16x + a (low) and + 8 (high)
          const uint2 lo2 = code_pair(widen2<DT>(xv[8 * x + i]), n2, r2, worst);
          const uint2 hi2 = code_pair(widen2<DT>(xv[8 * x + 4 + i]), n2, r2, worst);
          vc[4 * x + 2 * i * 64] = static_cast<uint8_t>(lo2.x + (hi2.x << 4));
          vc[4 * x + (2 * i + 1) * 64] = static_cast<uint8_t>(lo2.y + (hi2.y << 4));
        }
      } else {
        uint2 q[4];   // channels 32k + 8qq + 2i, + 1
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) q[qq] = code_pair(widen2<DT>(xv[4 * qq + i]), n2, r2, worst);
        vc[2 * i * 64] = static_cast<uint8_t>(q[0].x + (q[1].x << 2) + (q[2].x << 4) + (q[3].x << 6));
        vc[(2 * i + 1) * 64] = static_cast<uint8_t>(q[0].y + (q[1].y << 2) + (q[2].y << 4) + (q[3].y << 6));
      }
      flags |= (worst > kTieGuard ? 1u : 0u) << i;
    }
    if (vslow) flags = 0xfu;
    if (flags) value_bytes_fix<BITS, DT>(flags, Vs, t, k, lo, sc, vc);
  }
  // read before the barrier: once past it, thread 0 may refill this stage's refs
  const int slot = tile_ref[0], pp0 = tile_ref[1], pp1 = tile_ref[2];
  __syncthreads();
  char* rec0 = nullptr;
  char* rec1 = nullptr;
  if (slot < 0 || slot >= a.max_slots) {
    if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
  } else {
    if (pp0 >= 0 && pp0 < a.num_pages) rec0 = a.pages + (static_cast<long long>(pp0) * a.H + it.h) * F::kBytes;
    else if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp0);
    if (pp1 >= 0 && pp1 < a.num_pages) rec1 = a.pages + (static_cast<long long>(pp1) * a.H + it.h) * F::kBytes;
    else if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp1);
  }
  // ---- both staged records to their pages ----------------------------------
  constexpr int kChunks = F::kBytes / 16;
#pragma unroll
  for (int q = tid; q < 2 * kChunks; q += kThreads) {
    const bool p1 = q >= kChunks;
    char* rec = p1 ? rec1 : rec0;
    const int off = (q - (p1 ? kChunks : 0)) * 16;
    if (rec) *reinterpret_cast<uint4*>(rec + off) = *reinterpret_cast<const uint4*>((p1 ? st1 : st0) + off);
  }
}

// Copies the new rows bound for a ring: tokens [tb, T1) into rows t % mod. The
// first 16-byte chunk of each thread was loaded early (first); the rest are
// loaded four at a time before they are stored.
__device__ __forceinline__ void ring_copy(uint16_t* ring, int mod, int tb, int T1, const uint16_t* src_base,
                                          long long row_of_t0, int H, int h, uint4 first) {
  const int n = (T1 - tb) * 16;
  int q = threadIdx.x;
  if (q < n) reinterpret_cast<uint4*>(ring + static_cast<long long>((tb + q / 16) % mod) * kD)[q % 16] = first;
  q += kThreads;
  for (; q + 3 * kThreads < n; q += 4 * kThreads) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int qq = q + u * kThreads, t = tb + qq / 16;
      v[u] = reinterpret_cast<const uint4*>(row_ptr(src_base, row_of_t0 + t, H, h))[qq % 16];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int qq = q + u * kThreads, t = tb + qq / 16;
      reinterpret_cast<uint4*>(ring + static_cast<long long>(t % mod) * kD)[qq % 16] = v[u];
    }
  }
  for (; q < n; q += kThreads) {
    const int t = tb + q / 16;
    reinterpret_cast<uint4*>(ring + static_cast<long long>(t % mod) * kD)[q % 16] =
        reinterpret_cast<const uint4*>(row_ptr(src_base, row_of_t0 + t, H, h))[q % 16];
  }
}

// A ring item of a decode-like step, inlined in the kernel's loop: at most one
// value token per warp leaves the window and no key group mixes ring and new
// rows. The same steps as the ring item of other_item.
__device__ __forceinline__ bool ring_item_is_few(const AppendArgs& a, const Item& it) {
  if (it.j != 0) return false;
  const int Tv0 = max(0, it.T0 - a.R), Tv1 = max(0, it.T1 - a.R);
  const int vend = min(it.T0, Tv1);
  const int Tk0 = it.T0 & ~(kG - 1);
  return vend - Tv0 <= kThreads / 32 && !(Tk0 < it.T0 && Tk0 + kG <= it.T1);
}

template <int BITS>
__device__ __forceinline__ void ring_item_few(const AppendArgs& a, const Item& it) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = it.i, h = it.h, T0 = it.T0, T1 = it.T1, row0 = it.row0;
  const int slot = a.slot_ids ? a.slot_ids[i] : i;
  if (slot < 0 || slot >= a.max_slots) {
    if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
    return;
  }
  if (static_cast<long long>(a.bt_stride) * kP < T1) {
    if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, i);
    return;
  }
  Ctx c{&a, a.block_table + static_cast<long long>(i) * a.bt_stride, slot};
  uint16_t* kring = reinterpret_cast<uint16_t*>(a.kring) + slot * a.kring_slot + h * a.kring_head;
  uint16_t* vring = reinterpret_cast<uint16_t*>(a.vring) + slot * a.vring_slot + h * a.vring_head;
  const int Tk1 = T1 & ~(kG - 1);
  const int Tv0 = max(0, T0 - a.R), Tv1 = max(0, T1 - a.R);
  int* len_word = a.lens + slot * a.H + h;
  const int stored = *len_word;
  const int tv = Tv0 + warp, vend = min(T0, Tv1);
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
    return;
  }
  if (tv < vend) value_token_row<BITS>(c, h, tv, vraw, vpage);
  __syncthreads();
  ring_copy(kring, kG, kb, T1, a.k, static_cast<long long>(row0) - T0, a.H, h, kfirst);
  ring_copy(vring, a.R, vb, T1, a.v, static_cast<long long>(row0) - T0, a.H, h, vfirst);
  if (tid == 0) *len_word = T1;
  __syncthreads();
}

// Ring items and the tiles that are not whole new key groups.
template <int BITS>
__device__ __noinline__ void other_item(const AppendArgs& a, const Item it, uint8_t (*stage)[1536], const uint16_t** src,
                                       uint8_t* rows) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = it.i, h = it.h, j = it.j, T0 = it.T0, T1 = it.T1, row0 = it.row0;
  const int slot = a.slot_ids ? a.slot_ids[i] : i;
  if (slot < 0 || slot >= a.max_slots) {
    if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
    return;
  }
  if (static_cast<long long>(a.bt_stride) * kP < T1) {
    if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, i);
    return;
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
    // A decode step's few leaving tokens (one per warp at most) go by the token
    // path, their rows and pages loaded together with the stored length.
    constexpr int kW = kThreads / 32;
    const bool few = vend - Tv0 <= kW;
    uint2 vraw = make_uint2(0u, 0u);
    int vpage = 0;
    if (few && Tv0 + warp < vend) {
      vraw = *reinterpret_cast<const uint2*>(vring + static_cast<long long>((Tv0 + warp) % a.R) * kD + 4 * lane);
      vpage = c.bt_row[(Tv0 + warp) / kP];
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
      return;
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
    // Value tokens leaving the window, 64 at a time: every thread's loads of the
    // batch's ring rows (and of the pool pages they fall in) are in flight
    // together and land in shared memory (the item's free tile stage, as two
    // 32-row tiles in the layout of tile_prefetch); then each lane quantizes one
    // 32-channel group of one token per tile, as the tile path does, into the
    // token's page record in the pool.
    if (few) {
      if (Tv0 + warp < vend) value_token_row<BITS>(c, h, Tv0 + warp, vraw, vpage);
    } else {
      constexpr int kLeaveTiles = kStageBytes / kTileBytes;        // 2
      constexpr int kLeaveRows = kLeaveTiles * kG;                  // 64
      constexpr int kPer = kLeaveRows * (kD * 2 / 16) / kThreads;   // 16-byte chunks per thread
      __shared__ int bpage[kLeaveRows / kP + 1];
      for (int base = Tv0; base < vend; base += kLeaveRows) {
        const int cnt = min(kLeaveRows, vend - base);
        const int p_lo = base / kP, np = (base + cnt - 1) / kP - p_lo + 1;
        uint4 v[kPer];
#pragma unroll
        for (int x = 0; x < kPer; ++x) {
          const int q = tid + kThreads * x, r = q >> 4;
          v[x] = r < cnt ? reinterpret_cast<const uint4*>(vring + static_cast<long long>((base + r) % a.R) * kD)[q & 15]
                         : make_uint4(0u, 0u, 0u, 0u);
        }
        const int pg = tid < np ? c.bt_row[p_lo + tid] : 0;
        __syncthreads();   // the previous batch is quantized: the buffer is free
#pragma unroll
        for (int x = 0; x < kPer; ++x) {
          const int q = tid + kThreads * x, r = q >> 4;
          if (r < cnt) *reinterpret_cast<uint4*>(rows + (r >> 5) * kTileBytes + sw_off(r & 31, q & 15)) = v[x];
        }
        if (tid < np) bpage[tid] = pg;
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kLeaveTiles; ++u) {
          const int r = kG * u + 8 * warp + (lane & 7);
          if (r < cnt) {
            const int tok = base + r, pp = bpage[tok / kP - p_lo];
            if (pp >= 0 && pp < a.num_pages) {
              uint8_t* rec =
                  reinterpret_cast<uint8_t*>(a.pages) + (static_cast<long long>(pp) * a.H + h) * Rec<BITS>::kBytes;
              if (a.dtype == S4KV_BF16) value_lane<BITS, S4KV_BF16>(rows + u * kTileBytes, r & (kG - 1), tok, rec, lane >> 3);
              else value_lane<BITS, S4KV_F16>(rows + u * kTileBytes, r & (kG - 1), tok, rec, lane >> 3);
            } else {
              report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp);
            }
          }
        }
      }
    }
    __syncthreads();
    ring_copy(kring, kG, kb, T1, a.k, static_cast<long long>(row0) - T0, a.H, h, kfirst);
    ring_copy(vring, a.R, vb, T1, a.v, static_cast<long long>(row0) - T0, a.H, h, vfirst);
    if (tid == 0) *len_word = T1;
    __syncthreads();
  } else {
    const int tile = it.tile;
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
}

template <int BITS, int DT>
__global__ void __launch_bounds__(kThreads, kAppendCtas) append_kernel(AppendArgs a) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ int warp_tot[kThreads / 32];
  __shared__ const uint16_t* src[kG];
  int* pre = reinterpret_cast<int*>(dsm);   // [n + 1]
  int* seq = reinterpret_cast<int*>(dsm + seq_info_offset(a.n));
  int* cpre = reinterpret_cast<int*>(dsm + cost_prefix_offset(a.n));   // [n + 1]
  uint8_t* stages = dsm + prefix_bytes(a.n);
  uint8_t* staging = stages + kNumStages * kStageBytes;
  float* prm = reinterpret_cast<float*>(staging + kStagingBytes);

  if (!build_prefix(a, pre, warp_tot, seq, cpre)) return;
  // A CTA takes the items that start in its slice of the work line, in order;
  // whole new tiles are loaded kNumStages - 1 items ahead (one cp.async group per
  // item, empty for other items).
  const long long C = cpre[a.n];
  int item = item_from_cost(a, pre, seq, cpre, C * blockIdx.x / gridDim.x);
  const int total = item_from_cost(a, pre, seq, cpre, C * (blockIdx.x + 1) / gridDim.x);   // this CTA's end
  if (item >= total) return;
  constexpr int kAhead = kNumStages - 1;
  const int step = 1;
  Item i0 = item_of(a, pre, seq, item), i1;
  i1.fast = false;
  __shared__ int tile_refs[kNumStages][4];   // per stage: slot, pool pages of the tile's two records
  if (i0.fast) tile_prefetch(a, i0, stages, tile_refs[0]);
  cp_async_commit();
  if constexpr (kAhead == 2) {
    if (item + step < total) {
      i1 = item_of(a, pre, seq, item + step);
      if (i1.fast) tile_prefetch(a, i1, stages + kStageBytes, tile_refs[1]);
    }
    cp_async_commit();
  }
  int s = 0;
  while (item < total) {
    Item in;   // the item kAhead ahead
    in.fast = false;
    const int sn = s + kAhead >= kNumStages ? s + kAhead - kNumStages : s + kAhead;
    if (item + kAhead * step < total) {
      in = item_of(a, pre, seq, item + kAhead * step);
      if (in.fast) tile_prefetch(a, in, stages + sn * kStageBytes, tile_refs[sn]);
    }
    cp_async_commit();
    // One barrier before each item: the item's cp.async rows are in shared
    // memory, and the previous item is done with the staging buffer (a fast
    // tile's stage is refilled only kNumStages - 1 items later, past that
    // barrier).
    if (i0.fast) {
      cp_async_wait_prev();
      __syncthreads();
      fast_tile<BITS, DT>(a, i0, stages + s * kStageBytes, tile_refs[s], staging, prm);
    } else if (ring_item_is_few(a, i0)) {
      __syncthreads();
      ring_item_few<BITS>(a, i0);
    } else {
      __syncthreads();
      other_item<BITS>(a, i0, reinterpret_cast<uint8_t (*)[1536]>(staging), src, stages + s * kStageBytes);
    }
    if constexpr (kAhead == 2) {
      i0 = i1;
      i1 = in;
    } else {
      i0 = in;
    }
    item += step;
    s = s + 1 == kNumStages ? 0 : s + 1;
  }
  cp_async_wait_all();
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

int append_ctas_per_sm() { return kAppendCtas; }

cudaError_t launch_append(const AppendArgs& a, int grid, cudaStream_t st) {
  if (a.n <= 0 || grid <= 0) return cudaSuccess;
  if (a.n > kMaxSeqsPerCall) return cudaErrorInvalidValue;
  if (a.bits == 8) {
    const size_t smem = static_cast<size_t>(a.n + 1) * sizeof(int);
    const cudaError_t c = prefer_max_shared(reinterpret_cast<const void*>(append_fp8_kernel));
    if (c != cudaSuccess) return c;
    append_fp8_kernel<<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
  }
  const int smem = append_smem_bytes(a.n);
  void (*kern)(AppendArgs);
  if (a.bits == 2) kern = a.dtype == S4KV_BF16 ? append_kernel<2, S4KV_BF16> : append_kernel<2, S4KV_F16>;
  else kern = a.dtype == S4KV_BF16 ? append_kernel<4, S4KV_BF16> : append_kernel<4, S4KV_F16>;
  {
    const cudaError_t c = prefer_max_shared(reinterpret_cast<const void*>(kern));
    if (c != cudaSuccess) return c;
  }
  if (smem > 48 * 1024) {
    // raise the kernel's dynamic shared memory limit once per device and size
    static std::mutex lock;
    static int raised[kMaxAppendDevices][4] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxAppendDevices) return cudaErrorInvalidDevice;
    const int v = (a.bits == 2 ? 2 : 0) + (a.dtype == S4KV_BF16 ? 1 : 0);
    std::lock_guard<std::mutex> guard(lock);
    if (raised[dev][v] < smem) {
      const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      raised[dev][v] = smem;
    }
  }
  kern<<<grid, kThreads, smem, st>>>(a);
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
