// Device-side building blocks shared by the attention kernels (s4kv_decode.cu:
// decode attention and its merge; s4kv_mq.cu: multi-query attention): PTX
// helpers (mbarriers, bulk copies, mma.sync), the staged-record geometry, the
// unpacking of codes into MMA operands, the per-group decode arithmetic, the FP8
// page arithmetic, the cost-line work partition, the shared-memory layout, the
// partial and merge-descriptor workspace, and the host helpers that launch
// kernels. Internal to the library (not part of the public ABI); everything sits
// in an unnamed namespace, so each translation unit holds its own copy.
#pragma once

#include "s4kv_common.cuh"

#include <cuda_fp8.h>

namespace s4kv {
namespace {

// Worker warps per CTA of the tensor-core path and the CTAs per SM its
// register budget is sized for (a build-time tuning pair: 12 x 1 gives 168
// registers a thread; 8 x 2 gives 128). The FFMA path runs 8 warps, 1 CTA/SM.
#ifndef S4KV_DECODE_WARPS
#define S4KV_DECODE_WARPS 12
#endif
#ifndef S4KV_DECODE_MIN_CTAS
#define S4KV_DECODE_MIN_CTAS 1
#endif
template <int IMPL>
__host__ __device__ constexpr int warps_of() { return IMPL == 1 ? 8 : S4KV_DECODE_WARPS; }
constexpr int kStages = 2;
// A stage holds one key group: two page records, the second shifted by 64
// bytes so that equal offsets of the two records fall in different banks.
constexpr int kRecStride = kRec + 64;
constexpr int kStageBytes = kRecStride + kRec;
// Each warp owns one flat region: two stages in the main loop; in the tail one
// group's page records (or key-ring rows) at 0, then the group's value-ring rows
// at a stride of kVRow bytes (16 more than a row, so that the eight rows read by
// one ldmatrix fall in different banks), all staged by one batch of bulk copies.
constexpr int kVRow = kD * 2 + 16;
constexpr int kVoffRecs = 2 * kRecStride;                 // value rows after page records
constexpr int kRegion = kVoffRecs + kG * kVRow;           // 14976 bytes
// A tail group's n < 32 key-ring rows are staged beside its n value rows when
// they fit; otherwise the keys are read from the ring in global memory.
constexpr int kKringStageMax = kRegion / (kD * 2 + kVRow);
static_assert(kStages * kStageBytes <= kRegion, "two main-loop stages fit the region");
// The same strides for a record of BITS-bit codes (the 4-bit ones above are the largest).
template <int BITS> constexpr int kRecStrideB = Rec<BITS>::kBytes + 64;
template <int BITS> constexpr int kStageBytesB = kRecStrideB<BITS> + Rec<BITS>::kBytes;
template <int BITS> constexpr int kVoffRecsB = 2 * kRecStrideB<BITS>;
static_assert(kVoffRecs % 16 == 0 && kVRow % 16 == 0 && kRegion % 128 == 0, "bulk copy alignment");
static_assert(kKringStageMax >= 16 && kKringStageMax < kG, "key-ring staging bound");
constexpr int kPRow = 12;                       // row stride of the P tile (floats), conflict-free
constexpr int kNH = kMaxGroup;                  // head slots per kv head (GQA group <= 8)
constexpr long long kDrainNs = 1000000000LL;    // limit for draining copies after a timeout

// Phase timeline of every worker warp (tuning builds only, -DS4KV_DECODE_TRACE):
// 64-bit words per warp after the partials in the workspace.
#ifdef S4KV_DECODE_TRACE
constexpr int kTraceWords = 22;
#define S4KV_TRACE(...) __VA_ARGS__
#else
constexpr int kTraceWords = 0;
#define S4KV_TRACE(...)
#endif

// ---- PTX helpers -------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// 1-D bulk copy global -> shared (TMA), completing on `bar`, with an L2 cache
// policy for the bytes it reads.
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// L2 policy for data read once per launch (page records, ring rows): evicted
// first, so that what is reused (block tables, queries, partials) stays.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same, letting the thread sleep inside try_wait (up to 1 us a try) and reading
// the timer only every 64 tries: for waits that are routinely long.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, long long limit_ns) {
  if (limit_ns <= 0) return false;
  const unsigned long long t0 = global_ns();
  for (unsigned it = 1;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(1000u)
        : "memory");
    if (ok) return true;
    if ((it & 63u) == 0 && static_cast<long long>(global_ns() - t0) > limit_ns) return false;
  }
}

// Bounded wait: false once `limit_ns` has passed (limit 0: give up at once).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit_ns) {
  if (limit_ns <= 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (static_cast<long long>(global_ns() - t0) > limit_ns) return false;
  }
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lop_and_or(uint32_t x, uint32_t mask, uint32_t bits) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "r"(mask), "r"(bits));
  return r;
}

// 2-bit codes of one slice (odd = 0: positions 0, 1; odd = 1: positions 2, 3) of
// w as f16 subnormals: rows of the lower position come out at 1 (odd: 16) times
// n * 2^-24, rows of the upper position at 4 (odd: 64) times n * 2^-24.
__device__ __forceinline__ void unpack_crumbs_sub(uint32_t w, int odd, uint32_t (&a)[4]) {
  const uint32_t w8 = w >> 8;
  const uint32_t m0 = odd ? 0x00300030u : 0x00030003u, m1 = odd ? 0x00C000C0u : 0x000C000Cu;
  a[0] = w & m0;
  a[1] = w & m1;
  a[2] = w8 & m0;
  a[3] = w8 & m1;
}

// The same slice as exact integer codes: a 2-bit field at position p OR-ed into
// 1024.0 (0x6400) is 1024 + 4^p n, and (x - 1024) * 4^-p leaves n exactly.
__device__ __forceinline__ void unpack_crumbs(uint32_t w, int odd, uint32_t (&a)[4]) {
  const uint32_t kMagic = 0x64006400u;
  const uint32_t w8 = w >> 8;
  const uint32_t m0 = odd ? 0x00300030u : 0x00030003u, m1 = odd ? 0x00C000C0u : 0x000C000Cu;
  // 4^-p and -1024 * 4^-p for p = 2 odd, 2 odd + 1 (f16 bit patterns, exact)
  const uint16_t s0 = odd ? 0x2C00 : 0x3C00, s1 = odd ? 0x2400 : 0x3400;   // 1/16, 1/64 | 1, 1/4
  const uint16_t o0 = odd ? 0xD400 : 0xE400, o1 = odd ? 0xCC00 : 0xDC00;   // -64, -16 | -1024, -256
  const __half2 sc0 = __halves2half2(__ushort_as_half(s0), __ushort_as_half(s0));
  const __half2 sc1 = __halves2half2(__ushort_as_half(s1), __ushort_as_half(s1));
  const __half2 of0 = __halves2half2(__ushort_as_half(o0), __ushort_as_half(o0));
  const __half2 of1 = __halves2half2(__ushort_as_half(o1), __ushort_as_half(o1));
  const uint32_t x[4] = {lop_and_or(w, m0, kMagic), lop_and_or(w, m1, kMagic), lop_and_or(w8, m0, kMagic),
                         lop_and_or(w8, m1, kMagic)};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&x[i]), (i & 1) ? sc1 : sc0, (i & 1) ? of1 : of0);
    a[i] = *reinterpret_cast<const uint32_t*>(&r);
  }
}

// Eight nibbles n0..n7 of w to four f16x2 registers holding the exact integer
// codes (n0, n4), (n1, n5), (n2, n6), (n3, n7). OR-ing a nibble into the low
// mantissa bits of 1024.0 (0x6400) gives 1024 + n; a nibble at bits 4..7 gives
// 1024 + 16 n; subtracting (or scaling and subtracting) leaves n exactly.
// The same four registers as f16 subnormals, with no arithmetic: a nibble alone
// in the low mantissa bits of a zero exponent is the f16 value n * 2^-24, and a
// nibble at bits 4..7 is 16 n * 2^-24, both exact. An MMA over these operands
// yields 2^-24 times the code sum (rows of low nibbles) or 2^-20 times it (rows
// of high nibbles), and the caller multiplies that power of two back out.
__device__ __forceinline__ void unpack8_sub(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t w8 = w >> 8;
  a[0] = w & 0x000F000Fu;
  a[1] = w & 0x00F000F0u;
  a[2] = w8 & 0x000F000Fu;
  a[3] = w8 & 0x00F000F0u;
}
constexpr float kLowRows = 16777216.0f;   // 2^24: rows of low nibbles (A registers 0 and 2)
constexpr float kHighRows = 1048576.0f;   // 2^20: rows of high nibbles (A registers 1 and 3)

__device__ __forceinline__ void unpack8(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t kMagic = 0x64006400u;
  const uint32_t lo0 = lop_and_or(w, 0x000F000Fu, kMagic);
  const uint32_t hi0 = lop_and_or(w, 0x00F000F0u, kMagic);
  const uint32_t w8 = w >> 8;
  const uint32_t lo1 = lop_and_or(w8, 0x000F000Fu, kMagic);
  const uint32_t hi1 = lop_and_or(w8, 0x00F000F0u, kMagic);
  const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
  const __half2 k16th = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));  // 1/16
  const __half2 km64 = __halves2half2(__ushort_as_half(0xD400), __ushort_as_half(0xD400));   // -64
  __half2 r0 = __hsub2(*reinterpret_cast<const __half2*>(&lo0), k1024);
  __half2 r1 = __hfma2(*reinterpret_cast<const __half2*>(&hi0), k16th, km64);
  __half2 r2 = __hsub2(*reinterpret_cast<const __half2*>(&lo1), k1024);
  __half2 r3 = __hfma2(*reinterpret_cast<const __half2*>(&hi1), k16th, km64);
  a[0] = *reinterpret_cast<uint32_t*>(&r0);
  a[1] = *reinterpret_cast<uint32_t*>(&r1);
  a[2] = *reinterpret_cast<uint32_t*>(&r2);
  a[3] = *reinterpret_cast<uint32_t*>(&r3);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Exact small-integer to float: 2^23 + n has n in its low mantissa bits.
__device__ __forceinline__ float code_to_float(uint32_t n) {
  return __int_as_float(0x4B000000 | n) - 8388608.0f;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// 2^x with the SFU instruction (ex2.approx, relative error about 2^-22; -inf -> 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The running maximum of the online softmax is raised only when a score
// exceeds it by more than this many log2 units; probabilities then stay below
// 2^kLazy, and rescaling the accumulators becomes rare.
constexpr float kLazy = 6.0f;
// |q'| * sm_scale * log2(e) above which a key slice's q' also gets its low f16
// part: the rounding of f16(q') there would move a score by more than about
// 15 * 2^-12 * 0.25 = 1e-3 (log2 domain) per channel.
constexpr float kLoAbove = 0.25f;



// ---- per-segment context -------------------------------------------------------------
// A segment is one (sequence b, kv head h) pair: T tokens read by g query heads.
struct Seg {
  const char* pages;      // layer page region
  const int* bt;          // block-table row of b
  const uint16_t* kring;  // this (slot, head)'s key ring
  const uint16_t* vring;  // this (slot, head)'s value ring
  int H, h, T, Tk, Tv, R, dtype;
};

// Record of pool page `page` for this segment's kv head.
template <int BITS = 4>
__device__ __forceinline__ const char* rec_at(const Seg& sg, int page) {
  return sg.pages + (static_cast<long long>(page) * sg.H + sg.h) * Rec<BITS>::kBytes;
}

template <int BITS = 4>
__device__ __forceinline__ const char* rec_of(const Seg& sg, int logical_page) {
  return sg.pages + (static_cast<long long>(sg.bt[logical_page]) * sg.H + sg.h) * Rec<BITS>::kBytes;
}

// Online-softmax state of a warp in the "channel-quad" layout: lane l owns
// channels 4l..4l+3 of every head; m (log2 domain) and l are warp-uniform.
struct GenState {
  float m[kNH], l[kNH], o[kNH][4];
};

__device__ __forceinline__ void gen_init(GenState& s) {
#pragma unroll
  for (int h = 0; h < kNH; ++h) {
    s.m[h] = -INFINITY;
    s.l[h] = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) s.o[h][q] = 0.0f;
  }
}

// Softmax update for one chunk of up to 32 token scores z (lane = token; -inf
// for absent tokens). Writes p into ptile[token * kPRow + head].
__device__ __forceinline__ void gen_softmax(GenState& s, const float (&z)[kNH], float* ptile) {
  const int lane = threadIdx.x & 31;
  float p[kNH];
#pragma unroll
  for (int h = 0; h < kNH; ++h) {
    const float cm = warp_max(z[h]);
    const float mn = fmaxf(s.m[h], cm);
    const float alpha = ex2(s.m[h] - mn);   // 0 while the state is empty (m = -inf)
    p[h] = ex2(z[h] - mn);                   // absent tokens have z = -inf
    const float sum = warp_sum(p[h]);
    s.l[h] = s.l[h] * alpha + sum;
    s.m[h] = mn;
#pragma unroll
    for (int q = 0; q < 4; ++q) s.o[h][q] *= alpha;
  }
  *reinterpret_cast<float4*>(ptile + lane * kPRow) = make_float4(p[0], p[1], p[2], p[3]);
  *reinterpret_cast<float4*>(ptile + lane * kPRow + 4) = make_float4(p[4], p[5], p[6], p[7]);
  __syncwarp();
}

// Restored values of value token tau (page-local) for channels 4l..4l+3, from
// a page record in shared memory.
__device__ __forceinline__ void value_quad(const char* rec, int tau, int l, float (&v)[4]) {
  const int b = (tau & 7) >> 1, wv = tau >> 3, r = tau & 1;
  const int bt = wv ? (r ? 3 : 1) : (r ? 2 : 0);
  const int e = r + 2 * wv;
  const int mt = l >> 2, k = l >> 3, high = (l & 3) >> 1;
  const float s = *reinterpret_cast<const float*>(rec + kVm + ((2 * k) * 4 + b) * 16 + 4 * e);
  const float mn = *reinterpret_cast<const float*>(rec + kVm + ((2 * k + 1) * 4 + b) * 16 + 4 * e);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int a = 4 * (l & 1) + q;
    const uint32_t byte =
        static_cast<uint8_t>(rec[kVc + (mt >> 2) * 512 + (4 * a + b) * 16 + (mt & 3) * 4 + bt]);
    const uint32_t code = high ? (byte >> 4) : (byte & 15u);
    v[q] = fmaf(code_to_float(code), s, mn);
  }
}

__device__ __forceinline__ void ring_quad(const uint16_t* row, int l, int dtype, float (&v)[4]) {
  const uint2 r = *reinterpret_cast<const uint2*>(row + 4 * l);
  v[0] = widen16(static_cast<uint16_t>(r.x & 0xffff), dtype);
  v[1] = widen16(static_cast<uint16_t>(r.x >> 16), dtype);
  v[2] = widen16(static_cast<uint16_t>(r.y & 0xffff), dtype);
  v[3] = widen16(static_cast<uint16_t>(r.y >> 16), dtype);
}

__device__ __forceinline__ void gen_pv_token(GenState& s, const float (&v)[4], const float* prow,
                                             int g = kNH) {
  const float4 p0 = *reinterpret_cast<const float4*>(prow);
  const float4 p1 = *reinterpret_cast<const float4*>(prow + 4);
  const float p[kNH] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
  for (int h = 0; h < kNH; ++h)
    if (h < g)
#pragma unroll
      for (int q = 0; q < 4; ++q) s.o[h][q] = fmaf(p[h], v[q], s.o[h][q]);
}

// Tail chunk: tokens [32 grp, min(32 grp + 32, T)), past the last group whose
// keys and values are both quantized. `recs` holds the group's page records
// staged in shared memory (the second one only if it exists); q_s is the
// query block [8][128] fp32. Keys come from the records (t < Tk) or the key
// ring, values from the records (t < Tv) or the value ring; per token, CUDA
// cores, restored exactly as fmaf(code, scale, min).
__device__ void tail_chunk(const Seg& sg, int grp, GenState& s, float* ptile, const float* q_s,
                           const char* recs, float scale) {
  const int lane = threadIdx.x & 31;
  const int t0 = 32 * grp, n = min(32, sg.T - t0);
  float z[kNH];
#pragma unroll
  for (int h = 0; h < kNH; ++h) z[h] = lane < n ? 0.0f : -INFINITY;
  if (lane < n) {
    const int t = t0 + lane;
    if (t < sg.Tk) {
      const char* rec = recs + (lane >> 4) * kRecStride;
      const int tau = lane & 15, a = tau & 7, sh = (tau >> 3) * 4;
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
        const char* mrec = recs + (b >> 1) * kRecStride + kKm + (b & 1) * 16;
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
          const uint4 w4 = *reinterpret_cast<const uint4*>(rec + kKc + kh * 512 + 64 * a + 16 * b);
          const uint32_t wd[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int kq = 0; kq < 4; ++kq) {
            const int kk = 4 * kh + kq, c = 32 * b + 4 * kk;
            const float4 s4 = *reinterpret_cast<const float4*>(mrec + kk * 32);
            const float4 m4 = *reinterpret_cast<const float4*>(mrec + kk * 32 + 256);
            const uint32_t w = wd[kq];
            const float k0 = fmaf(code_to_float((w >> sh) & 15u), s4.x, m4.x);
            const float k1 = fmaf(code_to_float((w >> (16 + sh)) & 15u), s4.y, m4.y);
            const float k2 = fmaf(code_to_float((w >> (8 + sh)) & 15u), s4.z, m4.z);
            const float k3 = fmaf(code_to_float((w >> (24 + sh)) & 15u), s4.w, m4.w);
#pragma unroll
            for (int h = 0; h < kNH; ++h) {
              const float4 q4 = *reinterpret_cast<const float4*>(q_s + h * kD + c);
              z[h] = fmaf(q4.x, k0, fmaf(q4.y, k1, fmaf(q4.z, k2, fmaf(q4.w, k3, z[h]))));
            }
          }
        }
      }
    } else {
      const uint16_t* row = sg.kring + static_cast<long long>(t % kG) * kD;
#pragma unroll 1
      for (int c0 = 0; c0 < kD; c0 += 32) {   // four 16-byte loads in flight per step
        uint4 r4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) r4[i] = *reinterpret_cast<const uint4*>(row + c0 + 8 * i);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = c0 + 8 * i;
          const uint32_t rw[4] = {r4[i].x, r4[i].y, r4[i].z, r4[i].w};
          float kv[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            kv[2 * e] = widen16(static_cast<uint16_t>(rw[e] & 0xffff), sg.dtype);
            kv[2 * e + 1] = widen16(static_cast<uint16_t>(rw[e] >> 16), sg.dtype);
          }
#pragma unroll
          for (int h = 0; h < kNH; ++h) {
            const float4 qa = *reinterpret_cast<const float4*>(q_s + h * kD + c);
            const float4 qb = *reinterpret_cast<const float4*>(q_s + h * kD + c + 4);
            z[h] = fmaf(qa.x, kv[0], fmaf(qa.y, kv[1], fmaf(qa.z, kv[2], fmaf(qa.w, kv[3], z[h]))));
            z[h] = fmaf(qb.x, kv[4], fmaf(qb.y, kv[5], fmaf(qb.z, kv[6], fmaf(qb.w, kv[7], z[h]))));
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < kNH; ++h) z[h] *= scale;
  }
  gen_softmax(s, z, ptile);
  for (int tau0 = 0; tau0 < n; tau0 += 8) {   // eight tokens' loads in flight per step
    float v[8][4];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = t0 + tau0 + u;
      if (tau0 + u >= n) {
#pragma unroll
        for (int q = 0; q < 4; ++q) v[u][q] = 0.0f;
      } else if (t < sg.Tv) {
        value_quad(recs + ((tau0 + u) >> 4) * kRecStride, (tau0 + u) & 15, lane, v[u]);
      } else {
        ring_quad(sg.vring + static_cast<long long>(t % sg.R) * kD, lane, sg.dtype, v[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (tau0 + u < n) gen_pv_token(s, v[u], ptile + (tau0 + u) * kPRow);
  }
  __syncwarp();
}

// ---- FFMA path over one staged key group ---------------------------------------------
__device__ void ffma_group(const char* stage, GenState& s, float* ptile, float* qp, const float* q_s,
                           float scale) {
  const int lane = threadIdx.x & 31;
  // q'_hc = q_hc * s_c for the group, and beta_h = sum_c q_hc * min_c.
  float beta[kNH];
  {
    const char* mrec = stage + (lane >> 4) * kRecStride;
    const int off = kKm + (2 * (lane & 7) + ((lane & 15) >> 3)) * 16;
    const float4 s4 = *reinterpret_cast<const float4*>(mrec + off);
    const float4 m4 = *reinterpret_cast<const float4*>(mrec + off + 256);
#pragma unroll
    for (int h = 0; h < kNH; ++h) {
      const float4 q4 = *reinterpret_cast<const float4*>(q_s + h * kD + 4 * lane);
      *reinterpret_cast<float4*>(qp + h * kD + 4 * lane) =
          make_float4(q4.x * s4.x, q4.y * s4.y, q4.z * s4.z, q4.w * s4.w);
      beta[h] = warp_sum(fmaf(q4.x, m4.x, fmaf(q4.y, m4.y, fmaf(q4.z, m4.z, q4.w * m4.w))));
    }
  }
  __syncwarp();
  float z[kNH];
#pragma unroll
  for (int h = 0; h < kNH; ++h) z[h] = beta[h];
  {
    const char* rec = stage + (lane >> 4) * kRecStride;
    const int tau = lane & 15, a = tau & 7, sh = (tau >> 3) * 4;
#pragma unroll 1
    for (int b = 0; b < 4; ++b) {
#pragma unroll
      for (int kh = 0; kh < 2; ++kh) {
        const uint4 w4 = *reinterpret_cast<const uint4*>(rec + kKc + kh * 512 + 64 * a + 16 * b);
        const uint32_t wd[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) {
          const int c = 32 * b + 4 * (4 * kh + kq);
          const uint32_t w = wd[kq];
          const float f0 = code_to_float((w >> sh) & 15u);
          const float f1 = code_to_float((w >> (16 + sh)) & 15u);
          const float f2 = code_to_float((w >> (8 + sh)) & 15u);
          const float f3 = code_to_float((w >> (24 + sh)) & 15u);
#pragma unroll
          for (int h = 0; h < kNH; ++h) {
            const float4 q4 = *reinterpret_cast<const float4*>(qp + h * kD + c);
            z[h] = fmaf(q4.x, f0, fmaf(q4.y, f1, fmaf(q4.z, f2, fmaf(q4.w, f3, z[h]))));
          }
        }
      }
    }
  }
#pragma unroll
  for (int h = 0; h < kNH; ++h) z[h] *= scale;
  gen_softmax(s, z, ptile);
#pragma unroll 2
  for (int tau = 0; tau < 32; ++tau) {
    float v[4];
    value_quad(stage + (tau >> 4) * kRecStride, tau & 15, lane, v);
    gen_pv_token(s, v, ptile + tau * kPRow);
  }
  __syncwarp();
}

// ---- tensor-core path over one staged key group ----------------------------------------
struct MmaState {
  float o[8][4];     // O[16mt + gi (+8)][head 2ti (+1)]
  float bias[4];     // sum_t p_t * vmin_tk for head gi, group k (this lane's tokens)
  float m0, m1;      // running max of heads 2ti, 2ti+1 (log2 domain)
  float l0, l1;      // running sums over this lane's tokens
};

__device__ __forceinline__ void mma_init(MmaState& s) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) s.o[i][j] = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) s.bias[k] = 0.0f;
  s.m0 = s.m1 = -INFINITY;
  s.l0 = s.l1 = 0.0f;
}

// Scores of a staged key group (two page records): acc0 covers tokens 0..15,
// acc1 tokens 16..31 (rows gi, gi+8; columns heads 2ti, 2ti+1), without the
// min term. The B operand of channel slice kk is q' = q * s for head gi
// (channels 32 ti + 4 kk + 0..3). Returns beta = sum_c q_c * min_c of head gi.
// kSplit: q' also enters as the f16 rest of its f16 rounding (a second MMA per
// slice, accumulated apart and added at the end), about 22 significant bits in
// all; otherwise f16 q' alone. kPacked (GQA groups of at most 4 heads, with
// lanes of columns 4..7 holding the query of head gi - 4): columns 0..3 take
// f16(q') and columns 4..7 the rest of the same heads, so one MMA per slice
// carries both; the halves are added across lanes ti, ti ^ 2 at the end, and
// columns 4..7 then repeat heads 0..3.
template <bool kSplit, int BITS = 4, bool kPacked = false>
__device__ __forceinline__ float kscores_quant(const char* stage, const float (&q)[32], float (&acc0)[4],
                                               float (&acc1)[4], float lo_above) {
  (void)lo_above;   // (the split covers every slice)
  static_assert(kSplit || !kPacked, "the packed form is a form of the split");
  using F = Rec<BITS>;
  constexpr int RS = kRecStrideB<BITS>;
  const int lane = threadIdx.x & 31, ti = lane & 3;
  float beta = 0.0f;
  const char* mrec = stage + (ti >> 1) * RS + F::kKm + (ti & 1) * 16;
  // key code words of the two pages: 8 per lane (4-bit: one per slice kk) or 4
  // (2-bit: slices 2kp and 2kp+1 share word kp)
  uint32_t wa[8], wb[8];
  {
    const uint4 wa0 = *reinterpret_cast<const uint4*>(stage + F::kKc + lane * 16);
    const uint4 wb0 = *reinterpret_cast<const uint4*>(stage + RS + F::kKc + lane * 16);
    wa[0] = wa0.x; wa[1] = wa0.y; wa[2] = wa0.z; wa[3] = wa0.w;
    wb[0] = wb0.x; wb[1] = wb0.y; wb[2] = wb0.z; wb[3] = wb0.w;
    if constexpr (BITS == 4) {
      const uint4 wa1 = *reinterpret_cast<const uint4*>(stage + F::kKc + 512 + lane * 16);
      const uint4 wb1 = *reinterpret_cast<const uint4*>(stage + RS + F::kKc + 512 + lane * 16);
      wa[4] = wa1.x; wa[5] = wa1.y; wa[6] = wa1.z; wa[7] = wa1.w;
      wb[4] = wb1.x; wb[5] = wb1.y; wb[6] = wb1.z; wb[7] = wb1.w;
    }
  }
  // 2-bit: the odd slice of a word comes out 16x larger; its B operand is q'/16
  auto unpack = [&](const uint32_t (&ww)[8], int kk, uint32_t (&a)[4]) {
    if constexpr (BITS == 4) unpack8_sub(ww[kk], a);
    else unpack_crumbs_sub(ww[kk >> 1], kk & 1, a);
  };
  // q . min and q * scale two channels per instruction (fp32 pairs)
  float2 beta2 = make_float2(0.0f, 0.0f);
  float lo0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, lo1[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // split: scores of the rest
  // packed: -1 in lanes of columns 4..7 (they send q' - f16(q')), 0 elsewhere (f16(q'))
  const float neg = (kPacked && (lane >> 2) >= 4) ? -1.0f : 0.0f;
  const float2 neg2 = make_float2(neg, neg);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const float4 s4 = *reinterpret_cast<const float4*>(mrec + kk * 32);
    const float4 m4 = *reinterpret_cast<const float4*>(mrec + kk * 32 + 256);
    const float2 q01 = make_float2(q[4 * kk], q[4 * kk + 1]), q23 = make_float2(q[4 * kk + 2], q[4 * kk + 3]);
    beta2 = __ffma2_rn(q01, make_float2(m4.x, m4.y), beta2);
    beta2 = __ffma2_rn(q23, make_float2(m4.z, m4.w), beta2);
    const float bsc = (BITS == 2 && (kk & 1)) ? 0.0625f : 1.0f;
    const float2 x01 = __fmul2_rn(q01, make_float2(s4.x * bsc, s4.y * bsc));
    const float2 x23 = __fmul2_rn(q23, make_float2(s4.z * bsc, s4.w * bsc));
    if constexpr (!kSplit) {
      const uint32_t b0 = pack_f16x2(x01.x, x01.y);
      const uint32_t b1 = pack_f16x2(x23.x, x23.y);
      uint32_t a[4];
      unpack(wa, kk, a);
      mma16816(acc0, a, b0, b1);
      unpack(wb, kk, a);
      mma16816(acc1, a, b0, b1);
    } else if constexpr (kPacked) {
      // f16(q') in columns 0..3; in columns 4..7, q' - f16(q') (exact in fp32) rounded to f16
      const float2 r01 = __half22float2(__floats2half2_rn(x01.x, x01.y));
      const float2 r23 = __half22float2(__floats2half2_rn(x23.x, x23.y));
      const float2 y01 = __ffma2_rn(r01, neg2, x01), y23 = __ffma2_rn(r23, neg2, x23);
      const uint32_t b0 = pack_f16x2(y01.x, y01.y);
      const uint32_t b1 = pack_f16x2(y23.x, y23.y);
      uint32_t a[4];
      unpack(wa, kk, a);
      mma16816(acc0, a, b0, b1);
      unpack(wb, kk, a);
      mma16816(acc1, a, b0, b1);
    } else {
      const float x0 = x01.x, x1 = x01.y, x2 = x23.x, x3 = x23.y;
      const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&h01), b1 = *reinterpret_cast<const uint32_t*>(&h23);
      uint32_t a0[4], a1[4];
      unpack(wa, kk, a0);
      mma16816(acc0, a0, b0, b1);
      unpack(wb, kk, a1);
      mma16816(acc1, a1, b0, b1);
      // f16 rounding of q' dominates the score error where a key channel has a
      // wide scale (outliers), and the rounding of many ordinary channels adds
      // up too: every slice sends the rest q' - f16(q') through a second MMA
      // (about 22 significant bits in all).
      {
        const float2 r01 = __half22float2(h01), r23 = __half22float2(h23);
        const uint32_t c0 = pack_f16x2(x0 - r01.x, x1 - r01.y), c1 = pack_f16x2(x2 - r23.x, x3 - r23.y);
        mma16816(lo0, a0, c0, c1);
        mma16816(lo1, a1, c0, c1);
      }
    }
  }
  if constexpr (kSplit && !kPacked) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc0[j] += lo0[j];
      acc1[j] += lo1[j];
    }
  }
  if constexpr (kPacked) {   // head h's two halves sit in columns h and h + 4: lanes ti and ti ^ 2
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc0[j] += __shfl_xor_sync(0xffffffffu, acc0[j], 2);
      acc1[j] += __shfl_xor_sync(0xffffffffu, acc1[j], 2);
    }
  }
  // rows gi (tokens a) came out at 2^-24, rows gi + 8 at 2^-20 (4-bit) or 2^-22
  // (2-bit)
  constexpr float kHi = BITS == 4 ? kHighRows : 4194304.0f;
  acc0[0] *= kLowRows;
  acc0[1] *= kLowRows;
  acc0[2] *= kHi;
  acc0[3] *= kHi;
  acc1[0] *= kLowRows;
  acc1[1] *= kLowRows;
  acc1[2] *= kHi;
  acc1[3] *= kHi;
  beta = beta2.x + beta2.y;
  beta += __shfl_xor_sync(0xffffffffu, beta, 1);
  beta += __shfl_xor_sync(0xffffffffu, beta, 2);
  return beta;
}

__device__ __forceinline__ void mma16816_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_in_dtype(float lo, float hi, int dtype) {
  if (dtype == S4KV_BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  return pack_f16x2(lo, hi);
}

// Scores of key-ring tokens t0 .. t0 + n - 1 (n <= 31, t0 a multiple of 32, so
// ring rows 0 .. n - 1), raw keys times raw queries, exact products: the ring
// rows are the A operand as they are (lane ti reads channels 32 ti + 4 kk..+3,
// the channel order of the quantized path), q in the cache dtype is B.
__device__ __forceinline__ void kscores_ring(const uint16_t* kring, int n, const float (&q)[32],
                                             int dtype, float (&acc0)[4], float (&acc1)[4]) {
  const int lane = threadIdx.x & 31, gi = lane >> 2, ti = lane & 3;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    float (&acc)[4] = p ? acc1 : acc0;
    const int r0 = 16 * p + gi, r1 = r0 + 8;
#pragma unroll
    for (int half = 0; half < 2; ++half) {   // channels 32 ti + 16 half .. + 15
      uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0, y0 = x0, y1 = x0;
      if (r0 < n) {
        const uint4* src = reinterpret_cast<const uint4*>(kring + r0 * kD + 32 * ti + 16 * half);
        x0 = src[0];
        x1 = src[1];
      }
      if (r1 < n) {
        const uint4* src = reinterpret_cast<const uint4*>(kring + r1 * kD + 32 * ti + 16 * half);
        y0 = src[0];
        y1 = src[1];
      }
      const uint32_t xr[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const uint32_t yr[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const int kk = 4 * half + k4;
        const uint32_t a[4] = {xr[2 * k4], yr[2 * k4], xr[2 * k4 + 1], yr[2 * k4 + 1]};
        const uint32_t b0 = pack_in_dtype(q[4 * kk], q[4 * kk + 1], dtype);
        const uint32_t b1 = pack_in_dtype(q[4 * kk + 2], q[4 * kk + 3], dtype);
        if (dtype == S4KV_BF16) mma16816_bf16(acc, a, b0, b1);
        else mma16816(acc, a, b0, b1);
      }
    }
  }
}

// One 32-token key group (two page records in `stage`). q holds this lane's
// query values q[gi][32 ti + 4 kk + j] (fp32, zero for heads >= g).
template <bool kSplit, int BITS = 4, bool kPacked = false>
__device__ void mma_group(const char* stage, MmaState& s, float* ptile, const float (&q)[32],
                          float scale, float lo_above) {
  using F = Rec<BITS>;
  constexpr int RS = kRecStrideB<BITS>;
  const int lane = threadIdx.x & 31, gi = lane >> 2, ti = lane & 3;
  float acc0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const float beta = kscores_quant<kSplit, BITS, kPacked>(stage, q, acc0, acc1, lo_above);
  const float beta0 = __shfl_sync(0xffffffffu, beta, 8 * ti);       // head 2ti
  const float beta1 = __shfl_sync(0xffffffffu, beta, 8 * ti + 4);   // head 2ti+1
  // online softmax for heads 2ti (even entries) and 2ti+1 (odd entries), in the
  // log2 domain: z = (acc + beta) * scale
  const float bs0 = beta0 * scale, bs1 = beta1 * scale;
  float mx0 = fmaf(fmaxf(fmaxf(acc0[0], acc0[2]), fmaxf(acc1[0], acc1[2])), scale, bs0);
  float mx1 = fmaf(fmaxf(fmaxf(acc0[1], acc0[3]), fmaxf(acc1[1], acc1[3])), scale, bs1);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  if (__any_sync(0xffffffffu, mx0 > s.m0 + kLazy || mx1 > s.m1 + kLazy)) {
    const float mn0 = fmaxf(s.m0, mx0), mn1 = fmaxf(s.m1, mx1);
    const float al0 = ex2(s.m0 - mn0), al1 = ex2(s.m1 - mn1);
    s.m0 = mn0;
    s.m1 = mn1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s.o[i][0] *= al0;
      s.o[i][1] *= al1;
      s.o[i][2] *= al0;
      s.o[i][3] *= al1;
    }
    s.l0 *= al0;
    s.l1 *= al1;
    // bias belongs to head gi: its factor sits in lanes with ti = gi / 2
    const float a_even = __shfl_sync(0xffffffffu, al0, gi >> 1);
    const float a_odd = __shfl_sync(0xffffffffu, al1, gi >> 1);
    const float ag = (gi & 1) ? a_odd : a_even;
#pragma unroll
    for (int k = 0; k < 4; ++k) s.bias[k] *= ag;
  }
  {
    const float2 off = make_float2(bs0 - s.m0, bs1 - s.m1), sc2 = make_float2(scale, scale);
    const float2 z0 = __ffma2_rn(make_float2(acc0[0], acc0[1]), sc2, off);
    const float2 z1 = __ffma2_rn(make_float2(acc0[2], acc0[3]), sc2, off);
    const float2 z2 = __ffma2_rn(make_float2(acc1[0], acc1[1]), sc2, off);
    const float2 z3 = __ffma2_rn(make_float2(acc1[2], acc1[3]), sc2, off);
    const float p00 = ex2(z0.x), p01 = ex2(z0.y), p02 = ex2(z1.x), p03 = ex2(z1.y);
    const float p10 = ex2(z2.x), p11 = ex2(z2.y), p12 = ex2(z3.x), p13 = ex2(z3.y);
    s.l0 += (p00 + p02) + (p10 + p12);
    s.l1 += (p01 + p03) + (p11 + p13);
    *reinterpret_cast<float2*>(ptile + gi * kPRow + 2 * ti) = make_float2(p00, p01);
    *reinterpret_cast<float2*>(ptile + (gi + 8) * kPRow + 2 * ti) = make_float2(p02, p03);
    *reinterpret_cast<float2*>(ptile + (16 + gi) * kPRow + 2 * ti) = make_float2(p10, p11);
    *reinterpret_cast<float2*>(ptile + (24 + gi) * kPRow + 2 * ti) = make_float2(p12, p13);
  }
  __syncwarp();
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const char* rec = stage + p * RS;
    // p for tokens 2ti, 2ti+1, 2ti+8, 2ti+9 of this page, head gi
    const float pe0 = ptile[(16 * p + 2 * ti) * kPRow + gi];
    const float pe1 = ptile[(16 * p + 2 * ti + 1) * kPRow + gi];
    const float pe2 = ptile[(16 * p + 2 * ti + 8) * kPRow + gi];
    const float pe3 = ptile[(16 * p + 2 * ti + 9) * kPRow + gi];
    uint32_t b0[4], b1[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 s4 = *reinterpret_cast<const float4*>(rec + F::kVm + ((2 * k) * 4 + ti) * 16);
      const float4 m4 = *reinterpret_cast<const float4*>(rec + F::kVm + ((2 * k + 1) * 4 + ti) * 16);
      const float2 p01 = make_float2(pe0, pe1), p23 = make_float2(pe2, pe3);
      const float2 y01 = __fmul2_rn(p01, make_float2(s4.x, s4.y));
      const float2 y23 = __fmul2_rn(p23, make_float2(s4.z, s4.w));
      b0[k] = pack_f16x2(y01.x, y01.y);
      b1[k] = pack_f16x2(y23.x, y23.y);
      float2 u = __ffma2_rn(p01, make_float2(m4.x, m4.y), make_float2(s.bias[k], 0.0f));
      u = __ffma2_rn(p23, make_float2(m4.z, m4.w), u);
      s.bias[k] = u.x + u.y;
    }
    uint32_t vd[8];
    {
      const uint4 v0 = *reinterpret_cast<const uint4*>(rec + F::kVc + lane * 16);
      vd[0] = v0.x; vd[1] = v0.y; vd[2] = v0.z; vd[3] = v0.w;
      if constexpr (BITS == 4) {
        const uint4 v1 = *reinterpret_cast<const uint4*>(rec + F::kVc + 512 + lane * 16);
        vd[4] = v1.x; vd[5] = v1.y; vd[6] = v1.z; vd[7] = v1.w;
      }
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t a[4];
      // o rows accumulate at powers of two that mma_unscale removes
      if constexpr (BITS == 4) unpack8_sub(vd[mt], a);
      else unpack_crumbs_sub(vd[mt >> 1], mt & 1, a);
      mma16816(s.o[mt], a, b0[mt >> 1], b1[mt >> 1]);
    }
  }
  __syncwarp();
}

// Back from the main loop's operand scale (value codes as f16 subnormals) to
// true scale: channels 16 mt + gi were accumulated at 2^-24, channels 16 mt + gi + 8
// at 2^-20. Exact (powers of two).
// 2-bit codes: tiles mt even at 2^-24 (rows gi) and 2^-22 (rows gi + 8), odd
// tiles at 2^-20 and 2^-18.
template <int BITS = 4>
__device__ __forceinline__ void mma_unscale(MmaState& s) {
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const float lo = BITS == 4 ? kLowRows : (mt & 1) ? 1048576.0f : kLowRows;
    const float hi = BITS == 4 ? kHighRows : (mt & 1) ? 262144.0f : 4194304.0f;
    s.o[mt][0] *= lo;
    s.o[mt][1] *= lo;
    s.o[mt][2] *= hi;
    s.o[mt][3] *= hi;
  }
}


// Four 8x8 16-bit matrices, transposed: lane i gives the address of row i % 8
// of matrix i / 8; register j receives matrix j in the A-fragment layout.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&a)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr)
               : "memory");
}

// Four 8x8 16-bit matrices: lane i gives the address of row i % 8 of matrix
// i / 8; register j receives matrix j, thread T holding row T / 4, columns
// 2 (T % 4) and 2 (T % 4) + 1.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&a)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Tail group on the tensor-core path: tokens [t0, t1) = [32 grp, min(32 grp + 32, T)),
// folded into the MMA state. Key scores by MMA from the staged records (keys
// quantized) or the key-ring rows at `kring`; softmax as in mma_group, absent
// tokens at p = 0. P V by MMA, page by page: tokens below Tv from the staged
// records as in mma_group (p masked to those tokens); tokens from max(t0, Tv) on
// from the value-ring rows, which sit token-major at vrows + (t - t0) * kVRow.
// Those rows read transposed (ldmatrix .trans) are the A operand V^T; a row
// outside [max(t0, Tv), t1) reads the 16 zero bytes at `zero_s` instead. Ring
// values enter exactly in the cache dtype; p is split into a high and a low part
// in that dtype (two MMAs), keeping about 22 (f16) or 16 (bf16) bits: the most
// recent tokens often carry the largest weights.
template <int BITS = 4>
__device__ void tail_group(const Seg& sg, int grp, MmaState& s, float* ptile, const float (&q)[32],
                           const char* recs, const uint16_t* kring, const char* vrows, uint32_t zero_s,
                           float scale, int lim0, int lim1, unsigned long long* tt) {
  using F = Rec<BITS>;
  constexpr int RS = kRecStrideB<BITS>;
  const int lane = threadIdx.x & 31, gi = lane >> 2, ti = lane & 3;
  S4KV_TRACE(unsigned long long tq = global_ns();)
  const int t0 = 32 * grp, n = min(32, sg.T - t0), t1 = t0 + n;
  float acc0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  float beta = 0.0f;
  if (t0 + kG <= sg.Tk) beta = kscores_quant<true, BITS>(recs, q, acc0, acc1, kLoAbove / scale);
  else kscores_ring(kring, n, q, sg.dtype, acc0, acc1);
  const float bs0 = __shfl_sync(0xffffffffu, beta, 8 * ti) * scale;       // head 2ti
  const float bs1 = __shfl_sync(0xffffffffu, beta, 8 * ti + 4) * scale;   // head 2ti+1
  S4KV_TRACE(if (tt) { const unsigned long long x = global_ns(); tt[0] += x - tq; tq = x; })
  // z of this lane's tokens gi, gi+8, 16+gi, 24+gi for columns 2ti (limit lim0)
  // and 2ti+1 (limit lim1): a token t is visible to a column when t < its limit
  // (limits are at most T, so absent tokens are -inf too)
  float z[8];
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const float* acc = p ? acc1 : acc0;
    const int ta = t0 + 16 * p + gi, tb = ta + 8;
    z[4 * p + 0] = ta < lim0 ? fmaf(acc[0], scale, bs0) : -INFINITY;
    z[4 * p + 1] = ta < lim1 ? fmaf(acc[1], scale, bs1) : -INFINITY;
    z[4 * p + 2] = tb < lim0 ? fmaf(acc[2], scale, bs0) : -INFINITY;
    z[4 * p + 3] = tb < lim1 ? fmaf(acc[3], scale, bs1) : -INFINITY;
  }
  float mx0 = fmaxf(fmaxf(z[0], z[2]), fmaxf(z[4], z[6]));
  float mx1 = fmaxf(fmaxf(z[1], z[3]), fmaxf(z[5], z[7]));
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  if (__any_sync(0xffffffffu, mx0 > s.m0 + kLazy || mx1 > s.m1 + kLazy)) {
    const float mn0 = fmaxf(s.m0, mx0), mn1 = fmaxf(s.m1, mx1);
    // a column with no visible token so far keeps max -inf and an empty state
    const float al0 = mn0 == -INFINITY ? 1.0f : ex2(s.m0 - mn0);
    const float al1 = mn1 == -INFINITY ? 1.0f : ex2(s.m1 - mn1);
    s.m0 = mn0;
    s.m1 = mn1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s.o[i][0] *= al0;
      s.o[i][1] *= al1;
      s.o[i][2] *= al0;
      s.o[i][3] *= al1;
    }
    s.l0 *= al0;
    s.l1 *= al1;
    const float a_even = __shfl_sync(0xffffffffu, al0, gi >> 1);
    const float a_odd = __shfl_sync(0xffffffffu, al1, gi >> 1);
    const float ag = (gi & 1) ? a_odd : a_even;
#pragma unroll
    for (int k = 0; k < 4; ++k) s.bias[k] *= ag;
  }
  {
    float pz[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) pz[i] = z[i] == -INFINITY ? 0.0f : ex2(z[i] - ((i & 1) ? s.m1 : s.m0));
    s.l0 += (pz[0] + pz[2]) + (pz[4] + pz[6]);
    s.l1 += (pz[1] + pz[3]) + (pz[5] + pz[7]);
    *reinterpret_cast<float2*>(ptile + gi * kPRow + 2 * ti) = make_float2(pz[0], pz[1]);
    *reinterpret_cast<float2*>(ptile + (gi + 8) * kPRow + 2 * ti) = make_float2(pz[2], pz[3]);
    *reinterpret_cast<float2*>(ptile + (16 + gi) * kPRow + 2 * ti) = make_float2(pz[4], pz[5]);
    *reinterpret_cast<float2*>(ptile + (24 + gi) * kPRow + 2 * ti) = make_float2(pz[6], pz[7]);
  }
  __syncwarp();
  S4KV_TRACE(if (tt) { const unsigned long long x = global_ns(); tt[1] += x - tq; tq = x; })
  const int vt0 = max(t0, sg.Tv);
#pragma unroll 1
  for (int p = 0; p < 2; ++p) {
    const int tb = t0 + 16 * p;
    if (tb >= t1) break;
    // p of tokens 2ti, 2ti+1, 2ti+8, 2ti+9 of this page, head gi
    const float pe0 = ptile[(16 * p + 2 * ti) * kPRow + gi];
    const float pe1 = ptile[(16 * p + 2 * ti + 1) * kPRow + gi];
    const float pe2 = ptile[(16 * p + 2 * ti + 8) * kPRow + gi];
    const float pe3 = ptile[(16 * p + 2 * ti + 9) * kPRow + gi];
    if (tb < sg.Tv) {   // restored values: tokens tb .. Tv - 1 of this page
      const char* rec = recs + p * RS;
      const int nq = sg.Tv - tb;
      const bool q0 = 2 * ti < nq, q1 = 2 * ti + 1 < nq, q2 = 2 * ti + 8 < nq, q3 = 2 * ti + 9 < nq;
      uint32_t b0[4], b1[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 s4 = *reinterpret_cast<const float4*>(rec + F::kVm + ((2 * k) * 4 + ti) * 16);
        const float4 m4 = *reinterpret_cast<const float4*>(rec + F::kVm + ((2 * k + 1) * 4 + ti) * 16);
        b0[k] = pack_f16x2(q0 ? pe0 * s4.x : 0.0f, q1 ? pe1 * s4.y : 0.0f);
        b1[k] = pack_f16x2(q2 ? pe2 * s4.z : 0.0f, q3 ? pe3 * s4.w : 0.0f);
        float bk = s.bias[k];
        bk = q0 ? fmaf(pe0, m4.x, bk) : bk;
        bk = q1 ? fmaf(pe1, m4.y, bk) : bk;
        bk = q2 ? fmaf(pe2, m4.z, bk) : bk;
        bk = q3 ? fmaf(pe3, m4.w, bk) : bk;
        s.bias[k] = bk;
      }
      uint32_t vd[8];
      {
        const uint4 v0 = *reinterpret_cast<const uint4*>(rec + F::kVc + lane * 16);
        vd[0] = v0.x; vd[1] = v0.y; vd[2] = v0.z; vd[3] = v0.w;
        if constexpr (BITS == 4) {
          const uint4 v1 = *reinterpret_cast<const uint4*>(rec + F::kVc + 512 + lane * 16);
          vd[4] = v1.x; vd[5] = v1.y; vd[6] = v1.z; vd[7] = v1.w;
        }
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t a[4];   // exact integer codes: the state is at true scale here
        if constexpr (BITS == 4) unpack8(vd[mt], a);
        else unpack_crumbs(vd[mt >> 1], mt & 1, a);
        mma16816(s.o[mt], a, b0[mt >> 1], b1[mt >> 1]);
      }
    }
    if (tb + kP > vt0) {   // value-ring rows of this page
      // this lane's ldmatrix row: matrix j = lane / 8 (tokens +8 for j >= 2,
      // channels +8 for odd j), row lane % 8
      const int j = lane >> 3;
      const int row = 16 * p + (lane & 7) + 8 * (j >> 1);
      const bool present = t0 + row >= vt0 && t0 + row < t1;
      const uint32_t base = present ? smem_u32(vrows + row * kVRow + 16 * (j & 1)) : zero_s;
      const uint32_t step = present ? 32u : 0u;   // 16 channels further per tile
      if (sg.dtype == S4KV_BF16) {
        const uint32_t h0 = pack_bf16x2(pe0, pe1), h1 = pack_bf16x2(pe2, pe3);
        const uint32_t l0 = pack_bf16x2(pe0 - __uint_as_float(h0 << 16), pe1 - __uint_as_float(h0 & 0xffff0000u));
        const uint32_t l1 = pack_bf16x2(pe2 - __uint_as_float(h1 << 16), pe3 - __uint_as_float(h1 & 0xffff0000u));
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t a[4];
          ldsm_x4_trans(base + mt * step, a);
          mma16816_bf16(s.o[mt], a, h0, h1);
          mma16816_bf16(s.o[mt], a, l0, l1);
        }
      } else {
        const __half2 h0 = __floats2half2_rn(pe0, pe1), h1 = __floats2half2_rn(pe2, pe3);
        const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&h0), b1 = *reinterpret_cast<const uint32_t*>(&h1);
        const uint32_t l0 = pack_f16x2(pe0 - f0.x, pe1 - f0.y), l1 = pack_f16x2(pe2 - f1.x, pe3 - f1.y);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t a[4];
          ldsm_x4_trans(base + mt * step, a);
          mma16816(s.o[mt], a, b0, b1);
          mma16816(s.o[mt], a, l0, l1);
        }
      }
    }
  }
  __syncwarp();
  S4KV_TRACE(if (tt) { tt[2] += global_ns() - tq; })
}

// MMA state -> channel-quad state, through `scratch` (>= 1104 floats): O rows
// padded to 132 floats so the fragment writes are conflict-free.
__device__ void mma_to_gen(MmaState& s, GenState& g, float* scratch) {
  constexpr int kRow = kD + 4;
  const int lane = threadIdx.x & 31, gi = lane >> 2, ti = lane & 3;
  float* O = scratch;                   // [8][132]
  float* ML = scratch + kNH * kRow;     // m[8], l[8]
  float* BI = ML + 2 * kNH;             // bias[8 heads][4 groups]
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int c0 = 16 * mt + gi;
    O[(2 * ti) * kRow + c0] = s.o[mt][0];
    O[(2 * ti + 1) * kRow + c0] = s.o[mt][1];
    O[(2 * ti) * kRow + c0 + 8] = s.o[mt][2];
    O[(2 * ti + 1) * kRow + c0 + 8] = s.o[mt][3];
  }
  float bias[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    bias[k] = s.bias[k] + __shfl_xor_sync(0xffffffffu, s.bias[k], 1);
    bias[k] += __shfl_xor_sync(0xffffffffu, bias[k], 2);
  }
  BI[gi * 4 + ti] = ti == 0 ? bias[0] : ti == 1 ? bias[1] : ti == 2 ? bias[2] : bias[3];
  float l0 = s.l0, l1 = s.l1;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  if (gi == 0) {
    ML[2 * ti] = s.m0;
    ML[2 * ti + 1] = s.m1;
    ML[kNH + 2 * ti] = l0;
    ML[kNH + 2 * ti + 1] = l1;
  }
  __syncwarp();
#pragma unroll
  for (int h = 0; h < kNH; ++h) {
    g.m[h] = ML[h];
    g.l[h] = ML[kNH + h];
    const float bk = BI[h * 4 + (lane >> 3)];   // channels 4l..4l+3 lie in value group l / 8
    const float4 o4 = *reinterpret_cast<const float4*>(O + h * kRow + 4 * lane);
    g.o[h][0] = o4.x + bk;
    g.o[h][1] = o4.y + bk;
    g.o[h][2] = o4.z + bk;
    g.o[h][3] = o4.w + bk;
  }
  __syncwarp();
}

// ---- FP8 E4M3 pages on the tensor-core path --------------------------------------------
// A warp streams single page records (4 KiB) through three stages of its region.
constexpr int kFp8Stages = 3;
static_assert(kFp8Stages * Rec<8>::kBytes <= kRegion, "three FP8 stages fit the region");
static_assert(kFp8Stages <= 2 * kStages, "one mbarrier per FP8 stage");

// Two e4m3 bytes (low byte first) -> f16x2, exact (every E4M3 value is an f16 value).
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint32_t pair) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(pair), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// One FP8 page (16 tokens) folded into the state of head gi (m: running max in
// the log2 domain, l: this lane's running sum) and the output tiles s.o.
// Scores S = Q K^T take the GQA heads as the rows of the A operand (rows gi + 8
// are zero) and the page's tokens as the columns of two n8 tiles, so the scores
// a lane ends with (tokens 2ti, 2ti+1 and 2ti+8, 2ti+9 of head gi) are already
// the B operand of P V, which takes V^T (channels as rows) as A. Keys meet the
// query unscaled, so with q in f16 every product is exact; `scale` carries
// sm_scale * log2(e) * the key scale. With kMask (a sequence's last page),
// tokens from `nvalid` on are masked: their scores to -inf, their value
// operands to zero (their bytes are undefined, possibly NaN codes).
template <bool kMask>
__device__ __forceinline__ void fp8_page(const char* rec, MmaState& s, float& m, float& l,
                                         const uint32_t (&qa)[8][2], float scale, int nvalid) {
  const int lane = threadIdx.x & 31, ti = lane & 3;
  uint4 kw[4];
#pragma unroll
  for (int kp = 0; kp < 4; ++kp) kw[kp] = *reinterpret_cast<const uint4*>(rec + Rec<8>::kKc + kp * 512 + lane * 16);
  float s0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t w0 = (kk & 1) ? kw[kk >> 1].z : kw[kk >> 1].x;   // tokens gi | gi + 8, channels c_0, c_1
    const uint32_t w1 = (kk & 1) ? kw[kk >> 1].w : kw[kk >> 1].y;   // the same for c_2, c_3
    const uint32_t a[4] = {qa[kk][0], 0u, qa[kk][1], 0u};
    mma16816(s0, a, fp8x2_to_f16x2(w0 & 0xffffu), fp8x2_to_f16x2(w1 & 0xffffu));
    mma16816(s1, a, fp8x2_to_f16x2(w0 >> 16), fp8x2_to_f16x2(w1 >> 16));
  }
  float z[4] = {s0[0] * scale, s0[1] * scale, s1[0] * scale, s1[1] * scale};
  if (kMask) {
    z[0] = 2 * ti < nvalid ? z[0] : -INFINITY;
    z[1] = 2 * ti + 1 < nvalid ? z[1] : -INFINITY;
    z[2] = 2 * ti + 8 < nvalid ? z[2] : -INFINITY;
    z[3] = 2 * ti + 9 < nvalid ? z[3] : -INFINITY;
  }
  float mx = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  if (__any_sync(0xffffffffu, mx > m + kLazy)) {
    const float mn = fmaxf(m, mx);   // finite: every page holds a valid token
    const float al = ex2(m - mn);
    m = mn;
    l *= al;
    // output columns are heads 2ti and 2ti + 1: their factors sit in lanes 8ti and 8ti + 4
    const float al0 = __shfl_sync(0xffffffffu, al, 8 * ti);
    const float al1 = __shfl_sync(0xffffffffu, al, 8 * ti + 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s.o[i][0] *= al0;
      s.o[i][1] *= al1;
      s.o[i][2] *= al0;
      s.o[i][3] *= al1;
    }
  }
  float p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = ex2(z[i] - m);
  l += (p[0] + p[1]) + (p[2] + p[3]);
  const uint32_t b0 = pack_f16x2(p[0], p[1]), b1 = pack_f16x2(p[2], p[3]);
  uint4 vw[4];
#pragma unroll
  for (int kp = 0; kp < 4; ++kp) vw[kp] = *reinterpret_cast<const uint4*>(rec + Rec<8>::kVc + kp * 512 + lane * 16);
  uint32_t m01 = 0xffffffffu, m23 = 0xffffffffu;   // token halves of value registers 0, 1 and 2, 3
  if (kMask) {
    m01 = (2 * ti < nvalid ? 0x0000ffffu : 0u) | (2 * ti + 1 < nvalid ? 0xffff0000u : 0u);
    m23 = (2 * ti + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * ti + 9 < nvalid ? 0xffff0000u : 0u);
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const uint32_t w0 = (mt & 1) ? vw[mt >> 1].z : vw[mt >> 1].x;   // tokens 2ti, 2ti+1: channels +0 | +8
    const uint32_t w1 = (mt & 1) ? vw[mt >> 1].w : vw[mt >> 1].y;   // tokens 2ti+8, 2ti+9
    uint32_t a[4] = {fp8x2_to_f16x2(w0 & 0xffffu), fp8x2_to_f16x2(w0 >> 16), fp8x2_to_f16x2(w1 & 0xffffu),
                     fp8x2_to_f16x2(w1 >> 16)};
    if (kMask) {
      a[0] &= m01;
      a[1] &= m01;
      a[2] &= m23;
      a[3] &= m23;
    }
    mma16816(s.o[mt], a, b0, b1);
  }
}

// One FP8 page for 16 (query, head) columns of a multi-query call: the warp's
// columns are the 16 rows of the key-score A operand (rows gi and gi + 8), the
// page's tokens the columns of two n8 tiles, so each lane's scores (tokens
// 2ti, 2ti+1 | 2ti+8, 2ti+9 of columns gi and gi + 8) are the B operands of
// P V for the two n8 column tiles o[.][0] (columns 2ti, 2ti+1) and o[.][1]
// (columns 8 + 2ti, 9 + 2ti). m[r], l[r]: running max and this lane's sum of
// column row r (0: gi, 1: gi + 8). With kMask (the last pages), token tok0 + x
// is masked for a column from the column's causal limit on (limits never pass
// T), and the value operands of tokens from nvalid on are zeroed.
template <bool kMask>
__device__ __forceinline__ void fp8_page_mq(const char* rec, float (&o)[8][2][4], float (&m)[2], float (&l)[2],
                                            const uint32_t (&qa)[8][4], float scale, int tok0, int lim_lo,
                                            int lim_hi, int nvalid) {
  const int lane = threadIdx.x & 31, ti = lane & 3;
  uint4 kw[4];
#pragma unroll
  for (int kp = 0; kp < 4; ++kp) kw[kp] = *reinterpret_cast<const uint4*>(rec + Rec<8>::kKc + kp * 512 + lane * 16);
  float s0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t w0 = (kk & 1) ? kw[kk >> 1].z : kw[kk >> 1].x;
    const uint32_t w1 = (kk & 1) ? kw[kk >> 1].w : kw[kk >> 1].y;
    const uint32_t a[4] = {qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]};
    mma16816(s0, a, fp8x2_to_f16x2(w0 & 0xffffu), fp8x2_to_f16x2(w1 & 0xffffu));
    mma16816(s1, a, fp8x2_to_f16x2(w0 >> 16), fp8x2_to_f16x2(w1 >> 16));
  }
  float z[2][4] = {{s0[0] * scale, s0[1] * scale, s1[0] * scale, s1[1] * scale},
                   {s0[2] * scale, s0[3] * scale, s1[2] * scale, s1[3] * scale}};
  if (kMask) {
    const int tx[4] = {tok0 + 2 * ti, tok0 + 2 * ti + 1, tok0 + 2 * ti + 8, tok0 + 2 * ti + 9};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      z[0][x] = tx[x] < lim_lo ? z[0][x] : -INFINITY;
      z[1][x] = tx[x] < lim_hi ? z[1][x] : -INFINITY;
    }
  }
  float mx[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    mx[r] = fmaxf(fmaxf(z[r][0], z[r][1]), fmaxf(z[r][2], z[r][3]));
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
  }
  if (__any_sync(0xffffffffu, mx[0] > m[0] + kLazy || mx[1] > m[1] + kLazy)) {
    float al[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float mn = fmaxf(m[r], mx[r]);
      al[r] = mn == -INFINITY ? 1.0f : ex2(m[r] - mn);   // a column with nothing visible yet stays empty
      m[r] = mn;
      l[r] *= al[r];
    }
    // output columns 8ct + 2ti and 8ct + 2ti + 1 keep their state in lanes 8ti and 8ti + 4, row ct
#pragma unroll
    for (int ct = 0; ct < 2; ++ct) {
      const float a0 = __shfl_sync(0xffffffffu, al[ct], 8 * ti);
      const float a1 = __shfl_sync(0xffffffffu, al[ct], 8 * ti + 4);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][ct][0] *= a0;
        o[mt][ct][1] *= a1;
        o[mt][ct][2] *= a0;
        o[mt][ct][3] *= a1;
      }
    }
  }
  float p[2][4];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
#pragma unroll
    for (int x = 0; x < 4; ++x) p[r][x] = z[r][x] == -INFINITY ? 0.0f : ex2(z[r][x] - m[r]);
    l[r] += (p[r][0] + p[r][1]) + (p[r][2] + p[r][3]);
  }
  const uint32_t b00 = pack_f16x2(p[0][0], p[0][1]), b01 = pack_f16x2(p[0][2], p[0][3]);
  const uint32_t b10 = pack_f16x2(p[1][0], p[1][1]), b11 = pack_f16x2(p[1][2], p[1][3]);
  uint4 vw[4];
#pragma unroll
  for (int kp = 0; kp < 4; ++kp) vw[kp] = *reinterpret_cast<const uint4*>(rec + Rec<8>::kVc + kp * 512 + lane * 16);
  uint32_t m01 = 0xffffffffu, m23 = 0xffffffffu;
  if (kMask) {
    m01 = (2 * ti < nvalid ? 0x0000ffffu : 0u) | (2 * ti + 1 < nvalid ? 0xffff0000u : 0u);
    m23 = (2 * ti + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * ti + 9 < nvalid ? 0xffff0000u : 0u);
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const uint32_t w0 = (mt & 1) ? vw[mt >> 1].z : vw[mt >> 1].x;
    const uint32_t w1 = (mt & 1) ? vw[mt >> 1].w : vw[mt >> 1].y;
    uint32_t a[4] = {fp8x2_to_f16x2(w0 & 0xffffu), fp8x2_to_f16x2(w0 >> 16), fp8x2_to_f16x2(w1 & 0xffffu),
                     fp8x2_to_f16x2(w1 >> 16)};
    if (kMask) {
      a[0] &= m01;
      a[1] &= m01;
      a[2] &= m23;
      a[3] &= m23;
    }
    mma16816(o[mt][0], a, b00, b01);
    mma16816(o[mt][1], a, b10, b11);
  }
}

// ---- the kernel -------------------------------------------------------------------------
// Work partition. Every segment (b, h) costs one unit per key group of its main
// region, tail_cost units per tail chunk (or one unit if T = 0); the cost line
// of all segments is cut into equal contiguous slices, one per warp. A warp
// processes the units whose start lies in its slice. A segment inside one
// slice is written out directly; a segment cut by slice boundaries gets one
// partial (m, l, o) per overlapping warp, and the last of those to finish
// merges them. The weight of a tail chunk against a key group is a tuning
// knob (S4KV_OPT_TAIL_COST).
constexpr int kMinUnits = 4;

struct SegCost {
  int main_groups, tail_chunks;
  long long cost;
};

// FP8 pages have no residual: every 32-token chunk is a main group, the last
// one possibly partial.
template <int BITS = 4>
__device__ __forceinline__ SegCost seg_cost(int T, int R, int tail_cost) {
  SegCost c;
  if (T <= 0) {
    c.main_groups = c.tail_chunks = 0;
    c.cost = 1;
    return c;
  }
  if constexpr (BITS == 8) {
    c.main_groups = (T + kG - 1) / kG;
    c.tail_chunks = 0;
    c.cost = c.main_groups;
    return c;
  }
  const int Tk = T & ~(kG - 1), Tv = max(0, T - R);
  const int t_main = min(Tk, Tv) & ~(kG - 1);
  c.main_groups = t_main / kG;
  c.tail_chunks = (T - t_main + kG - 1) / kG;
  c.cost = c.main_groups + static_cast<long long>(tail_cost) * c.tail_chunks;
  return c;
}

template <int W>
struct Smem {
  alignas(128) uint8_t region[W][kRegion];
  alignas(16) float ptile[W][32 * kPRow];
  alignas(8) uint64_t bar[W][2 * kStages];   // per warp: full barriers; a team leader also its empty barriers
};
static_assert(sizeof(Smem<8>) % 16 == 0 && sizeof(Smem<12>) % 16 == 0,
              "shared layout must keep 16-byte alignment");

// FFMA path: per-warp query block and q' buffer; the tensor-core path keeps the
// query in registers.
template <int IMPL>
__host__ __device__ constexpr size_t extra_bytes() {
  return IMPL == 1 ? sizeof(float) * warps_of<1>() * 2 * kNH * kD : 0;
}
// Offset of the cost prefix array (int64 [B + 1]) in dynamic shared memory.
template <int IMPL>
__host__ __device__ constexpr size_t prefix_offset() {
  return (sizeof(Smem<warps_of<IMPL>()>) + extra_bytes<IMPL>() + 15) / 16 * 16;
}

// Floats of one partial result: O [g][128], then (m, l) per head, padded so
// every partial starts 16-byte aligned.
__host__ __device__ constexpr long long partial_floats(int g) { return static_cast<long long>(g) * kD + 4 * kNH; }

// Workspace: [two partials per worker warp of the grid][merge descriptors][trace].
// Descriptor (b, h) = (partial slot of the first contributor, contributors), as
// int32 x 2 packed in one int64; 0 contributors: nothing to merge. It is written
// by the warp whose slice holds the segment's first cost unit.
__host__ __device__ constexpr long long meta_words(int B, int H) { return (static_cast<long long>(B) * H + 1) / 2 * 2; }
__device__ __forceinline__ long long* meta_of(const DecodeArgs& a) {
  return reinterpret_cast<long long*>(a.ws + 2LL * a.grid_warps * partial_floats(a.pcols));
}

// Largest warp w with slice start r(w) = w * C / n <= x.
__device__ __forceinline__ int owner_of(long long x, long long C, int n) {
  int w = static_cast<int>((x * n) / C);
  while (w + 1 < n && ((w + 1) * C) / n <= x) ++w;
  while (w > 0 && (w * C) / n > x) --w;
  return w;
}

__device__ __forceinline__ void store_out(const DecodeArgs& a, long long row, int lane, float4 y) {
  const long long idx = row * kD + 4 * lane;
  if (a.out_dtype == S4KV_F32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + idx) = y;
  } else if (a.out_dtype == S4KV_F16) {
    const __half2 lo = __floats2half2_rn(y.x, y.y), hi = __floats2half2_rn(y.z, y.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(a.out) + idx) = u;
  } else {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(y.x, y.y), hi = __floats2bfloat162_rn(y.z, y.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + idx) = u;
  }
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Merge kernels: warps per CTA, and contributors loaded per round.
constexpr int kMergeWarps = 4;
constexpr int kMC = 8;

// Grants `kernel` the dynamic shared memory it needs (once per size increase).
cudaError_t grant_smem(void (*kernel)(DecodeArgs), size_t need, size_t* granted) {
  if (need <= *granted) return cudaSuccess;
  if (*granted == 0) {
    const cudaError_t c = prefer_max_shared(reinterpret_cast<const void*>(kernel));
    if (c != cudaSuccess) return c;
  }
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(need));
  if (e != cudaSuccess) {
    cudaGetLastError();   // leave no error behind for the caller's next CUDA call
    return e;
  }
  *granted = need;
  return cudaSuccess;
}

// Programmatic-dependent launch of a merge kernel right behind the attention kernel.
cudaError_t launch_merge(void (*kernel)(DecodeArgs), const DecodeArgs& a, long long items, int grid, cudaStream_t st) {
  if (items == 0) return cudaSuccess;
  const cudaError_t c = prefer_max_shared(reinterpret_cast<const void*>(kernel));
  if (c != cudaSuccess) return c;
  long long blocks = (items + kMergeWarps - 1) / kMergeWarps;
  if (blocks > 4LL * grid) blocks = 4LL * grid;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(32 * kMergeWarps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace
}  // namespace s4kv
