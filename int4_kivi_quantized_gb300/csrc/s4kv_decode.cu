// Read side of the cache: paged decode attention over the int4 history plus
// the full-precision residual ("4.4 KV Cache 量化", section 2: P = softmax(QK^T
// / sqrt d), output PV; section 3.2: residual and history both take part).
//
// One kernel per call, every warp an independent worker. The (sequence, kv head)
// segments are laid end to end on a cost line (one unit per 32-token key group,
// more per tail chunk) that is cut into one contiguous slice per warp. A warp
// streams its key groups through a two-stage ring in shared memory: both page
// records of a group (3 KiB each: codes and fp32 metadata of one kv head)
// arrive by 1-D bulk TMA, guarded by an mbarrier with a bounded wait. Nothing
// restored goes back to HBM ("给 KV cache 减肥", section 3.1: restore when the
// query reads):
//  * tensor-core path: the per-channel key scale is folded into the query
//    (q'_c = q_c s_c, one f16x2 operand per 16-channel slice) and the key min
//    into a per-head bias; nibbles are unpacked to f16 with the magic-number
//    method (integer OR into the mantissa of 1024.0, then subtract) and fed to
//    mma.sync m16n8k16 with tokens as rows and GQA heads as columns. The value
//    side folds the per-token scale into the probabilities (p'_t = p_t s_tk) and
//    the value min into a per-head, per-group bias, with channels as rows.
//  * FFMA path: the same staging with CUDA-core arithmetic, for comparison.
// Tokens past the last group quantized for both keys and values (at most
// R + 31) go through a per-token path that reads the rings. A segment inside
// one warp's slice is written directly; a segment split between warps leaves
// one (m, l, o) partial per warp and the last warp to finish merges them with
// the log-sum-exp rule.

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
// Multi-query over KIVI pages: the column count (nq g) from which each key group is
// restored once per team rather than folded into every warp's columns (measured on
// Llama-3.1-8B shapes: folding is 1.75x faster at 32 columns, restoring 1.2x at 64).
#ifndef S4KV_MQ_RESTORE_MIN_COLS
#define S4KV_MQ_RESTORE_MIN_COLS 64
#endif
// ... and from which the restored group feeds tcgen05 (mqt_kernel) instead of
// mma.sync: not by default (one group in flight per CTA, slower as built).
#ifndef S4KV_MQ_TC_MIN_COLS
#define S4KV_MQ_TC_MIN_COLS 1000
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
template <bool kSplit, int BITS = 4>
__device__ __forceinline__ float kscores_quant(const char* stage, const float (&q)[32], float (&acc0)[4],
                                               float (&acc1)[4], float lo_above) {
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
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const float4 s4 = *reinterpret_cast<const float4*>(mrec + kk * 32);
    const float4 m4 = *reinterpret_cast<const float4*>(mrec + kk * 32 + 256);
    beta = fmaf(q[4 * kk], m4.x, fmaf(q[4 * kk + 1], m4.y,
           fmaf(q[4 * kk + 2], m4.z, fmaf(q[4 * kk + 3], m4.w, beta))));
    const float bsc = (BITS == 2 && (kk & 1)) ? 0.0625f : 1.0f;
    if constexpr (!kSplit) {
      const uint32_t b0 = pack_f16x2(q[4 * kk] * s4.x * bsc, q[4 * kk + 1] * s4.y * bsc);
      const uint32_t b1 = pack_f16x2(q[4 * kk + 2] * s4.z * bsc, q[4 * kk + 3] * s4.w * bsc);
      uint32_t a[4];
      unpack(wa, kk, a);
      mma16816(acc0, a, b0, b1);
      unpack(wb, kk, a);
      mma16816(acc1, a, b0, b1);
    } else {
      const float x0 = q[4 * kk] * s4.x * bsc, x1 = q[4 * kk + 1] * s4.y * bsc;
      const float x2 = q[4 * kk + 2] * s4.z * bsc, x3 = q[4 * kk + 3] * s4.w * bsc;
      const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&h01), b1 = *reinterpret_cast<const uint32_t*>(&h23);
      uint32_t a0[4], a1[4];
      unpack(wa, kk, a0);
      mma16816(acc0, a0, b0, b1);
      unpack(wb, kk, a1);
      mma16816(acc1, a1, b0, b1);
      // A wide-scale (outlier) channel makes |q'| large, and f16 rounding of q'
      // then dominates the score's error: a 16-channel slice with such a channel
      // sends the rest q' - f16(q') through a second MMA (about 22 bits).
      if (__any_sync(0xffffffffu, fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3))) > lo_above * bsc)) {
        const float2 r01 = __half22float2(h01), r23 = __half22float2(h23);
        const uint32_t c0 = pack_f16x2(x0 - r01.x, x1 - r01.y), c1 = pack_f16x2(x2 - r23.x, x3 - r23.y);
        mma16816(acc0, a0, c0, c1);
        mma16816(acc1, a1, c0, c1);
      }
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
template <bool kSplit, int BITS = 4>
__device__ void mma_group(const char* stage, MmaState& s, float* ptile, const float (&q)[32],
                          float scale, float lo_above) {
  using F = Rec<BITS>;
  constexpr int RS = kRecStrideB<BITS>;
  const int lane = threadIdx.x & 31, gi = lane >> 2, ti = lane & 3;
  float acc0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const float beta = kscores_quant<kSplit, BITS>(stage, q, acc0, acc1, lo_above);
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
    const float off0 = bs0 - s.m0, off1 = bs1 - s.m1;
    const float p00 = ex2(fmaf(acc0[0], scale, off0)), p01 = ex2(fmaf(acc0[1], scale, off1));
    const float p02 = ex2(fmaf(acc0[2], scale, off0)), p03 = ex2(fmaf(acc0[3], scale, off1));
    const float p10 = ex2(fmaf(acc1[0], scale, off0)), p11 = ex2(fmaf(acc1[1], scale, off1));
    const float p12 = ex2(fmaf(acc1[2], scale, off0)), p13 = ex2(fmaf(acc1[3], scale, off1));
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
      b0[k] = pack_f16x2(pe0 * s4.x, pe1 * s4.y);
      b1[k] = pack_f16x2(pe2 * s4.z, pe3 * s4.w);
      s.bias[k] = fmaf(pe0, m4.x, fmaf(pe1, m4.y, fmaf(pe2, m4.z, fmaf(pe3, m4.w, s.bias[k]))));
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


template <int IMPL, int BITS>
__global__ void __launch_bounds__(32 * warps_of<IMPL>(), IMPL != 1 ? S4KV_DECODE_MIN_CTAS : 1)
    decode_kernel(DecodeArgs a) {
  static_assert(BITS == 4 || IMPL != 1, "the FFMA path reads 4-bit records");
  using F = Rec<BITS>;
  constexpr int RS = kRecStrideB<BITS>;
  constexpr int kWarps = warps_of<IMPL>();
  constexpr int kThreads = 32 * kWarps;
  using SmemT = Smem<kWarps>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmemT& sm = *reinterpret_cast<SmemT*>(smem_raw);
  long long* pre = reinterpret_cast<long long*>(smem_raw + prefix_offset<IMPL>());   // [B + 1]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* st0 = sm.region[warp];
  uint8_t* st1 = sm.region[warp] + kStageBytesB<BITS>;
  uint64_t* bar = sm.bar[warp];
  float* ptile = sm.ptile[warp];
  float* q_s = reinterpret_cast<float*>(smem_raw + sizeof(SmemT)) + warp * 2 * kNH * kD;   // FFMA path
  float* qp = q_s + kNH * kD;   // FFMA path only

  constexpr int kNS = BITS == 8 ? kFp8Stages : kStages;   // stages of the main loop
  if (lane == 0) {
    for (int i = 0; i < kNS; ++i) mbar_init(&bar[i], 1);
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __shared__ __align__(16) uint4 zero16;   // ldmatrix source of absent value-ring rows
  if (tid == 0) zero16 = make_uint4(0u, 0u, 0u, 0u);
  const uint32_t zero_s = smem_u32(&zero16);
  // cost prefix over sequences: sequence b owns H segments of seg_cost(T_b)
  {
    long long carry = 0;
    __shared__ long long wt[kWarps];
    for (int base = 0; base < a.B; base += kThreads) {
      const int b = base + tid;
      const long long cnt = b < a.B ? a.H * seg_cost<BITS>(a.seq_lens[b], a.R, a.tail_cost).cost : 0;
      long long x = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) wt[warp] = x;
      __syncthreads();
      long long before = carry, total = 0;
      for (int q = 0; q < kWarps; ++q) {
        if (q < warp) before += wt[q];
        total += wt[q];
      }
      if (b < a.B) pre[b] = before + x - cnt;
      __syncthreads();
      carry += total;
    }
    if (tid == 0) pre[a.B] = carry;
    __syncthreads();
  }
  const long long C = pre[a.B];
  int n_act = static_cast<int>(gridDim.x) * kWarps;
  if (a.max_warps > 0 && a.max_warps < n_act) n_act = a.max_warps;
  {
    // at least kMinUnits of work per warp: fewer partials on small problems
    const long long cap = (C + kMinUnits - 1) / kMinUnits;
    if (cap < n_act) n_act = static_cast<int>(cap);
  }
  // merge_kernel may be scheduled now; it waits for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int gw = blockIdx.x * kWarps + warp;
  if (gw >= n_act) return;
  const long long r0 = gw * C / n_act, r1 = (gw + 1) * C / n_act;
  // trace words: 0 start, 1 end, 2..5 phase times (prologue, main, tail, finalize), 6 segments,
  // 7 main groups, 8..10 tail parts (scores, softmax, PV), 11 tail groups, 12 main-loop waits,
  // 13 tail waits, 14 partial store + counter, 15 merges' time, 16 merges, 17 contributors
  // merged, 18 merge waits, 19 proxy fence, 20 fold, 21 output stores + counter reset
  S4KV_TRACE(unsigned long long tr[kTraceWords] = {};
             tr[0] = global_ns();
             int wslot = 12;
             unsigned long long tmark = tr[0];
             auto tlap = [&](int slot) { const unsigned long long t = global_ns(); tr[slot] += t - tmark; tmark = t; };)

  uint32_t phase = 0, pend = 0;   // per-stage wait parity and copies in flight (bit per stage)
  const uint64_t once = policy_evict_first();
  bool aborted = false;
  auto issue = [&](int s, int lp0, int np, const Seg& sg) {
    fence_proxy_async();   // earlier generic accesses of the buffer come first
    __syncwarp();
    if (lane == 0) {
      uint8_t* dst = s ? st1 : st0;
      mbar_expect_tx(&bar[s], np * kRec);
      for (int i = 0; i < np; ++i) bulk_load_hint(dst + i * kRecStride, rec_of(sg, lp0 + i), kRec, &bar[s], once);
    }
    pend |= 1u << s;
  };
  // both records of one key group, pool pages p0 and p1, into stage s
  auto issue_pp = [&](int s, int p0, int p1, const Seg& sg) {
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) {
      uint8_t* dst = s ? st1 : st0;
      mbar_expect_tx(&bar[s], 2 * F::kBytes);
      bulk_load_hint(dst, rec_at<BITS>(sg, p0), F::kBytes, &bar[s], once);
      bulk_load_hint(dst + RS, rec_at<BITS>(sg, p1), F::kBytes, &bar[s], once);
    }
    pend |= 1u << s;
  };
  auto wait = [&](int s) -> bool {
    S4KV_TRACE(const unsigned long long tw = global_ns();)
    const bool got = mbar_wait(&bar[s], (phase >> s) & 1u, aborted ? 0 : a.wait_ns);
    S4KV_TRACE(tr[wslot] += global_ns() - tw;)
    if (!got) return false;
    phase ^= 1u << s;
    pend &= ~(1u << s);
    return true;
  };
  auto fail = [&](long long where) {   // bounded wait ran out: drain, then go on without compute
    if (lane == 0) report(a.status, S4KV_ERR_DEVICE_TIMEOUT, S4KV_DEV_TIMEOUT, static_cast<int>(where));
    aborted = true;
    for (int s = 0; s < kNS; ++s) {
      if ((pend >> s) & 1u) {
        mbar_wait(&bar[s], (phase >> s) & 1u, kDrainNs);
        phase ^= 1u << s;
        pend &= ~(1u << s);
      }
    }
  };

  // first segment touching this slice
  int b;
  {
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  SegCost sc = seg_cost<BITS>(a.seq_lens[b], a.R, a.tail_cost);
  int h = static_cast<int>((r0 - pre[b]) / sc.cost);
  long long seg_start = pre[b] + h * sc.cost;

  while (seg_start < r1) {
    S4KV_TRACE(tr[6] += 1;)
    const long long seg_end = seg_start + sc.cost;
    const int T = max(a.seq_lens[b], 0);
    const long long lo = max(r0, seg_start) - seg_start, hi = min(r1, seg_end) - seg_start;
    const bool own = lo == 0 && hi == sc.cost;
    // main groups and tail chunks whose cost position starts inside [lo, hi)
    const int nm = sc.main_groups;
    const int u0 = static_cast<int>(lo < nm ? lo : nm), u1 = static_cast<int>(hi < nm ? hi : nm);
    int c0 = 0, c1 = 0;
    if (sc.tail_chunks > 0 && hi > nm) {
      c0 = static_cast<int>(lo > nm ? (lo - nm + a.tail_cost - 1) / a.tail_cost : 0);
      const long long cc = (hi - nm + a.tail_cost - 1) / a.tail_cost;
      c1 = static_cast<int>(cc < sc.tail_chunks ? cc : sc.tail_chunks);
    }
    const int slot = a.slot_ids ? a.slot_ids[b] : b;
    const bool slot_ok = slot >= 0 && slot < a.max_slots;
    const bool table_ok = static_cast<long long>(a.bt_stride) * kP >= T;
    // the segment's independent global reads are issued together: the cache's
    // length, the queries (tensor-core path) and the block-table entries
    const int lens_v = slot_ok ? a.lens[slot * a.H + h] : 0;
    float fp8_ks = 1.0f, fp8_vs = 1.0f;   // FP8 pages: the head's key and value scales
    if constexpr (BITS == 8) {
      fp8_ks = a.fp8_scale[h];
      fp8_vs = a.fp8_scale[a.H + h];
    }
    const uint16_t* qrow = a.q + (static_cast<long long>(b) * a.Hq + h * a.g) * kD;
    uint4 qraw[4];   // tensor-core path: this lane's query words, q[gi][32 ti .. 32 ti + 31]
    if constexpr (IMPL != 1) {
      const int gi = lane >> 2, ti = lane & 3;
#pragma unroll
      for (int i = 0; i < 4; ++i) qraw[i] = make_uint4(0u, 0u, 0u, 0u);
      if (gi < a.g && slot_ok && T > 0) {
        const uint4* src = reinterpret_cast<const uint4*>(qrow + gi * kD + 32 * ti);
#pragma unroll
        for (int i = 0; i < 4; ++i) qraw[i] = src[i];
      }
    }
    Seg sg;
    sg.pages = a.pages;
    sg.bt = a.block_table + static_cast<long long>(b) * a.bt_stride;
    sg.kring = reinterpret_cast<const uint16_t*>(a.kring) + (slot_ok ? slot : 0) * a.kring_slot + h * a.kring_head;
    sg.vring = reinterpret_cast<const uint16_t*>(a.vring) + (slot_ok ? slot : 0) * a.vring_slot + h * a.vring_head;
    sg.H = a.H;
    sg.h = h;
    sg.T = T;
    sg.Tk = T & ~(kG - 1);
    sg.Tv = max(0, T - a.R);
    sg.R = a.R;
    sg.dtype = a.dtype;
    bool valid = slot_ok && T > 0;
    bool bad = false;
    if (valid && table_ok && (u1 > u0 || c1 > c0)) {
      // every page this warp will read must be inside the pool
      const int p_lo = u1 > u0 ? 2 * u0 : 2 * (nm + c0);
      const int p_hi = min(c1 > c0 ? 2 * (nm + c1) : 2 * u1, (T + kP - 1) / kP);
      for (int base = p_lo; base < p_hi; base += 32 * 8) {   // eight loads in flight per lane
        int pp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int lp = base + 32 * k + lane;
          pp[k] = lp < p_hi ? sg.bt[lp] : 0;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (base + 32 * k + lane < p_hi && (pp[k] < 0 || pp[k] >= a.num_pages)) {
            bad = true;
            report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp[k]);
          }
        }
      }
    }
    if (!slot_ok) {
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
    } else if (lens_v != T || T > a.max_seq_len) {
      valid = false;
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, b);
    } else if (!table_ok) {
      valid = false;
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, b);
    }
    valid = valid && !__any_sync(0xffffffffu, bad) && !aborted;
    GenState gs;
    if (valid) {
      const int n = u1 - u0;
      float qv[32];   // tensor-core path: q[gi][32 ti + x], fp32
      if constexpr (IMPL != 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // heads >= g hold zero words, which widen to 0.0f
          const uint32_t w[4] = {qraw[i].x, qraw[i].y, qraw[i].z, qraw[i].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            qv[8 * i + 2 * j] = widen16(static_cast<uint16_t>(w[j] & 0xffff), a.dtype);
            qv[8 * i + 2 * j + 1] = widen16(static_cast<uint16_t>(w[j] >> 16), a.dtype);
          }
        }
        MmaState ms;
        mma_init(ms);
        S4KV_TRACE(tr[7] += n; tlap(2); wslot = 12;)
        bool ok = true;
        if constexpr (BITS == 8) {
          // pages pg0 .. pg1 - 1 of the slice (the last unit may hold one page, or a partial one)
          const int pg0 = 2 * u0, pg1 = min(2 * u1, (T + kP - 1) / kP), np = pg1 - pg0;
          uint32_t qa[8][2];   // A operand, row gi: head gi's query in f16, channels c_0 c_1 | c_2 c_3 of slice kk
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            qa[kk][0] = pack_f16x2(qv[4 * kk], qv[4 * kk + 1]);
            qa[kk][1] = pack_f16x2(qv[4 * kk + 2], qv[4 * kk + 3]);
          }
          const float zscale = a.sm_scale_log2 * fp8_ks;
          uint8_t* region = sm.region[warp];
          // pool pages pg0 + 32 k + lane, held one batch of 32 ahead of the copies
          auto page_of = [&](int k) {
            const int lp = pg0 + 32 * k + lane;
            return lp < pg1 ? sg.bt[lp] : 0;
          };
          int curp = page_of(0), nxtp = page_of(1), cur_k = 0;
          auto issue_page = [&](int st, int i) {   // i = 0, 1, 2, ... in order
            if ((i >> 5) != cur_k) {
              curp = nxtp;
              ++cur_k;
              nxtp = page_of(cur_k + 1);
            }
            const int pp = __shfl_sync(0xffffffffu, curp, i & 31);
            fence_proxy_async();   // earlier generic reads of the stage come first
            __syncwarp();
            if (lane == 0) {
              mbar_expect_tx(&bar[st], Rec<8>::kBytes);
              bulk_load_hint(region + st * Rec<8>::kBytes, rec_at<8>(sg, pp), Rec<8>::kBytes, &bar[st], once);
            }
            pend |= 1u << st;
          };
          for (int i = 0; i < np && i < kFp8Stages; ++i) issue_page(i, i);
          float m = -INFINITY, l = 0.0f;
          int st = 0;
          for (int i = 0; i < np; ++i) {
            if (!wait(st)) {
              ok = false;
              break;
            }
            const char* rec = reinterpret_cast<const char*>(region + st * Rec<8>::kBytes);
            const int nvalid = T - kP * (pg0 + i);
            if (nvalid < kP) fp8_page<true>(rec, ms, m, l, qa, zscale, nvalid);
            else fp8_page<false>(rec, ms, m, l, qa, zscale, kP);
            if (i + kFp8Stages < np) issue_page(st, i + kFp8Stages);
            st = st + 1 == kFp8Stages ? 0 : st + 1;
          }
          // into the MMA state's form (heads 2ti, 2ti + 1 per lane; sums in lanes gi = 0)
          l += __shfl_xor_sync(0xffffffffu, l, 1);
          l += __shfl_xor_sync(0xffffffffu, l, 2);
          const int ti = lane & 3;
          ms.m0 = __shfl_sync(0xffffffffu, m, 8 * ti);
          ms.m1 = __shfl_sync(0xffffffffu, m, 8 * ti + 4);
          const float l0 = __shfl_sync(0xffffffffu, l, 8 * ti), l1 = __shfl_sync(0xffffffffu, l, 8 * ti + 4);
          ms.l0 = lane < 4 ? l0 : 0.0f;
          ms.l1 = lane < 4 ? l1 : 0.0f;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) ms.o[mt][e] *= fp8_vs;
          S4KV_TRACE(tlap(3);)
        } else {
          // Pool pages of main groups u0 + 32 k + lane (two per group), held in
          // registers one batch of 32 groups ahead of the copies that need them.
          auto load_batch = [&](int k, int& x0, int& x1) {
            const int jj = u0 + 32 * k + lane;
            x0 = x1 = 0;
            if (jj < u1) {
              x0 = sg.bt[2 * jj];
              x1 = sg.bt[2 * jj + 1];
            }
          };
          int cur0, cur1, nxt0, nxt1, cur_k = 0;
          load_batch(0, cur0, cur1);
          load_batch(1, nxt0, nxt1);
          auto issue_group = [&](int s, int j) {   // j = 0, 1, 2, ... in order
            if ((j >> 5) != cur_k) {
              cur0 = nxt0;
              cur1 = nxt1;
              ++cur_k;
              load_batch(cur_k + 1, nxt0, nxt1);
            }
            const int p0 = __shfl_sync(0xffffffffu, cur0, j & 31);
            const int p1 = __shfl_sync(0xffffffffu, cur1, j & 31);
            issue_pp(s, p0, p1, sg);
          };
          for (int j = 0; j < n && j < kStages; ++j) issue_group(j, j);
          for (int j = 0; j < n; ++j) {
            const int s = j & 1;
            if (!wait(s)) { ok = false; break; }
            mma_group<IMPL == 2, BITS>(reinterpret_cast<const char*>(s ? st1 : st0), ms, ptile, qv,
                                       a.sm_scale_log2, kLoAbove / a.sm_scale_log2);
            if (j + kStages < n) issue_group(s, j + kStages);
          }
          mma_unscale<BITS>(ms);
          S4KV_TRACE(tlap(3);)
          unsigned long long* ttail = nullptr;   // tail phase counters (tracing builds)
          // pool pages of the first 16 tail groups: lane i holds logical page 2 (nm + c0) + i
          int tpg = 0;
          {
            const int lp = 2 * (nm + c0) + lane;
            if (c1 > c0 && lp < min(2 * (nm + c1), (T + kP - 1) / kP)) tpg = sg.bt[lp];
          }
          S4KV_TRACE(ttail = tr + 8; wslot = 13;)
          // Tail groups, one batch of bulk copies each into the warp's region: the
          // page records (keys and, where values are quantized, values) or the
          // key-ring rows, then the value-ring rows, one copy per row by the row's lane.
          for (int c = c0; ok && c < c1; ++c) {
            const int grp = nm + c;
            const int t0 = 32 * grp, t1 = min(t0 + kG, T);
            const bool kquant = t0 + kG <= sg.Tk;
            const bool vrec = t0 < sg.Tv;
            const bool kring_staged = !kquant && !vrec && t1 - t0 <= kKringStageMax;
            const int np = (t0 + kP < T) ? 2 : 1;
            const int vt0 = max(t0, sg.Tv);
            const int nv = max(0, t1 - vt0);
            const int voff = kring_staged ? (t1 - t0) * kD * 2 : kVoffRecsB<BITS>;
            uint32_t bytes = nv * kD * 2;
            if (vrec) bytes += np * F::kBytes;
            else if (kquant) bytes += np * (F::kKm + 512);
            if (kring_staged) bytes += (t1 - t0) * kD * 2;
            const int tp0 = __shfl_sync(0xffffffffu, tpg, (2 * (c - c0)) & 31);
            const int tp1 = __shfl_sync(0xffffffffu, tpg, (2 * (c - c0) + 1) & 31);
            fence_proxy_async();   // earlier generic accesses of the region come first
            __syncwarp();
            if (lane == 0) {
              mbar_expect_tx(&bar[0], bytes);
              if (vrec || kquant) {
                const bool held = c - c0 < 16;
                const char* r0 = held ? rec_at<BITS>(sg, tp0) : rec_of<BITS>(sg, 2 * grp);
                const char* r1 = np < 2 ? r0 : held ? rec_at<BITS>(sg, tp1) : rec_of<BITS>(sg, 2 * grp + 1);
                // whole records, or only the key codes and key metadata when no value is quantized
                const uint32_t rb = vrec ? F::kBytes : F::kKm + 512;
                bulk_load_hint(st0, r0, rb, &bar[0], once);
                if (np == 2) bulk_load_hint(st0 + RS, r1, rb, &bar[0], once);
              }
              if (kring_staged) bulk_load_hint(st0, sg.kring, (t1 - t0) * kD * 2, &bar[0], once);
            }
            __syncwarp();
            if (lane < nv) {
              const int t = vt0 + lane;
              bulk_load_hint(st0 + voff + (t - t0) * kVRow, sg.vring + static_cast<long long>(t % sg.R) * kD, kD * 2,
                             &bar[0], once);
            }
            pend |= 1u;
            if (!wait(0)) {
              ok = false;
              break;
            }
            tail_group<BITS>(sg, grp, ms, ptile, qv, reinterpret_cast<const char*>(st0),
                       kring_staged ? reinterpret_cast<const uint16_t*>(st0) : sg.kring,
                       reinterpret_cast<const char*>(st0 + voff), zero_s, a.sm_scale_log2, T, T, ttail);
            S4KV_TRACE(tr[11] += 1;)
          }
        }
        if (ok) mma_to_gen(ms, gs, reinterpret_cast<float*>(st0));
        else {
          fail(b);
          gen_init(gs);
        }
        S4KV_TRACE(tlap(4);)
      } else {
        gen_init(gs);
        // query block for the FFMA path: lane l writes channels 4l..4l+3
        for (int j = 0; j < kNH; ++j) {
          float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          if (j < a.g) ring_quad(qrow + j * kD, lane, a.dtype, v);
          *reinterpret_cast<float4*>(q_s + j * kD + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
        }
        __syncwarp();
        for (int j = 0; j < n && j < kStages; ++j) issue(j, 2 * (u0 + j), 2, sg);
        for (int j = 0; j < n; ++j) {
          const int s = j & 1;
          if (!wait(s)) {
            fail(b);
            gen_init(gs);
            break;
          }
          ffma_group(reinterpret_cast<const char*>(s ? st1 : st0), gs, ptile, qp, q_s, a.sm_scale_log2);
          if (j + kStages < n) issue(s, 2 * (u0 + j + kStages), 2, sg);
        }
      }
      if constexpr (IMPL == 1) {
        // tail chunks: page records (when any of their keys or values are
        // quantized) staged in stage 0
        for (int c = c0; c < c1 && !aborted; ++c) {
          const int grp = nm + c;
          const int np = (32 * grp + kP < T) ? 2 : 1;
          issue(0, 2 * grp, np, sg);
          if (!wait(0)) {
            fail(b);
            gen_init(gs);
            break;
          }
          tail_chunk(sg, grp, gs, ptile, q_s, reinterpret_cast<const char*>(st0), a.sm_scale_log2);
        }
      }
    } else {
      gen_init(gs);
    }

    // ---- output, or the partial that merge_kernel combines ----
    if (seg_start >= r0 && lane == 0) {   // this warp holds the segment's first unit: its merge descriptor
      int ncon = 0;
      if (!own && slot_ok) ncon = owner_of(seg_end - 1, C, n_act) - gw + 1;
      const long long first = 2LL * gw + (seg_start <= r0 ? 0 : 1);
      meta_of(a)[static_cast<long long>(b) * a.H + h] =
          static_cast<long long>(static_cast<unsigned>(first)) | (static_cast<long long>(ncon) << 32);
    }
    if (own || !slot_ok) {
#pragma unroll
      for (int j = 0; j < kNH; ++j) {
        if (j < a.g) {
          const float inv = gs.l[j] > 0.0f ? 1.0f / gs.l[j] : 0.0f;
          store_out(a, static_cast<long long>(b) * a.Hq + h * a.g + j, lane,
                    make_float4(gs.o[j][0] * inv, gs.o[j][1] * inv, gs.o[j][2] * inv, gs.o[j][3] * inv));
        }
      }
    } else {
      S4KV_TRACE(const unsigned long long tf0 = global_ns();)
      const int k = seg_start <= r0 ? 0 : 1;
      const long long part_floats = partial_floats(a.pcols);
      float* P = a.ws + (2LL * gw + k) * part_floats;
#pragma unroll
      for (int j = 0; j < kNH; ++j) {
        if (j < a.g) {
          *reinterpret_cast<float4*>(P + j * kD + 4 * lane) =
              make_float4(gs.o[j][0], gs.o[j][1], gs.o[j][2], gs.o[j][3]);
          if (lane == 0) {
            P[a.pcols * kD + 2 * j] = gs.m[j];
            P[a.pcols * kD + 2 * j + 1] = gs.l[j];
          }
        }
      }
      S4KV_TRACE(tr[14] += global_ns() - tf0;)
    }

    S4KV_TRACE(tlap(5);)
    // next segment
    seg_start = seg_end;
    if (++h == a.H) {
      h = 0;
      if (++b >= a.B) break;
      sc = seg_cost<BITS>(a.seq_lens[b], a.R, a.tail_cost);
    }
  }
  if (pend) fail(-1);   // never expected: every issued copy is waited for
  S4KV_TRACE({
    tr[1] = global_ns();
    if (lane == 0) {
      unsigned long long* out = reinterpret_cast<unsigned long long*>(meta_of(a) + meta_words(a.B, a.H)) +
                                static_cast<long long>(gw) * kTraceWords;
      for (int i = 0; i < kTraceWords; ++i) out[i] = tr[i];
    }
  })
}

// ---- merge of split segments ---------------------------------------------------------
// One warp per (segment, query head). It reads the segment's merge descriptor
// and skips segments written directly (inside one warp's slice, or an invalid
// slot); otherwise it combines the partials of the segment's contributors by
// the log-sum-exp rule, eight contributors at a time: their (m, l) pairs
// (lane = contributor) and rows are loaded together, then weighed and summed.
constexpr int kMergeWarps = 4;
constexpr int kMC = 8;

__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(DecodeArgs a) {
  S4KV_TRACE(const unsigned long long tm_start = global_ns();)
  asm volatile("griddepcontrol.wait;" ::: "memory");   // decode_kernel has completed; its writes are visible
  S4KV_TRACE(const unsigned long long tm_go = global_ns(); unsigned long long tm_seg = 0, tm_ld = 0;)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long* desc = meta_of(a);
  const long long items = static_cast<long long>(a.B) * a.H * a.g;
  const long long pf = partial_floats(a.pcols);
  for (long long it = static_cast<long long>(blockIdx.x) * kMergeWarps + warp; it < items;
       it += static_cast<long long>(gridDim.x) * kMergeWarps) {
    const int j = static_cast<int>(it % a.g);
    const long long bh = it / a.g;
    const long long d = __ldcg(desc + bh);
    const int nc = static_cast<int>(d >> 32);
    if (nc <= 0) continue;   // inside one slice, or an invalid slot: written by decode_kernel
    S4KV_TRACE(tm_seg = global_ns();)
    // contributor 0 is the descriptor's slot; contributor i >= 1 is the warp i
    // places on, slot 0 (the segment is the first piece of its slice)
    const long long first = static_cast<long long>(static_cast<unsigned>(d & 0xffffffffLL));
    auto part = [&](int i) -> const float* {
      return a.ws + (i == 0 ? first : (first & ~1LL) + 2LL * i) * pf;
    };
    float M = -INFINITY, L = 0.0f;
    float4 O = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int i0 = 0; i0 < nc; i0 += kMC) {
      const int nch = min(kMC, nc - i0);
      const float* W = part(i0 + (lane < nch ? lane : 0)) + a.pcols * kD + 2 * j;
      const float mi = lane < nch ? __ldcg(W) : -INFINITY;
      const float li = lane < nch ? __ldcg(W + 1) : 0.0f;
      float4 r[kMC];
#pragma unroll
      for (int u = 0; u < kMC; ++u)
        r[u] = u < nch ? __ldcg(reinterpret_cast<const float4*>(part(i0 + u) + j * kD + 4 * lane))
                       : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      S4KV_TRACE(if (!tm_ld) tm_ld = global_ns() + static_cast<unsigned long long>(r[kMC - 1].x == 12345.0f);)
      const float mn = fmaxf(M, warp_max(mi));
      const bool live = mn != -INFINITY;   // all partials empty so far: nothing to weigh
      const float ao = live ? ex2(M - mn) : 1.0f;
      const float wi = live ? ex2(mi - mn) : 0.0f;
      L = fmaf(L, ao, warp_sum(wi * li));
      O = make_float4(O.x * ao, O.y * ao, O.z * ao, O.w * ao);
#pragma unroll
      for (int u = 0; u < kMC; ++u) {
        const float w = __shfl_sync(0xffffffffu, wi, u);   // 0 for absent contributors
        O = make_float4(fmaf(w, r[u].x, O.x), fmaf(w, r[u].y, O.y), fmaf(w, r[u].z, O.z), fmaf(w, r[u].w, O.w));
      }
      M = mn;
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    store_out(a, static_cast<long long>(bh / a.H) * a.Hq + (bh % a.H) * a.g + j, lane,
              make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
  }
  S4KV_TRACE({
    // after the decode warps' words: (wait released, descriptor read, loads landed, end) of merge warp i
    const long long mw = static_cast<long long>(blockIdx.x) * kMergeWarps + warp;
    if (lane == 0 && mw < a.grid_warps) {
      unsigned long long* out = reinterpret_cast<unsigned long long*>(meta_of(a) + meta_words(a.B, a.H)) +
                                static_cast<long long>(a.grid_warps) * kTraceWords + 4 * mw;
      out[0] = tm_go;
      out[1] = tm_seg;
      out[2] = tm_ld;
      out[3] = global_ns();
    }
    (void)tm_start;
  })
}

// ---- multi-query attention: a chunk of query tokens per sequence ------------------------
// Causal attention of the last nq <= 16 tokens of every sequence (a chunk of a
// chunked prefill, or the tokens a speculative step verifies) over the length-T
// state after the chunk was appended: query i, at position T - nq + i, sees
// tokens 0 .. T - nq + i. Column c = i * g + j pairs query token i with head j
// of the kv head. A team of tw = ceil(nq g / 8) warps works on one slice of the
// cost line: its leader stages each key group once for the whole team (full
// barriers), every warp runs the decode arithmetic on its own 8 columns and
// then marks the stage free (empty barriers, one arrival per warp). Main groups
// need no mask (nq <= R puts them below every column's limit); tail groups
// take each column's limit.
template <int BITS>
__global__ void __launch_bounds__(32 * S4KV_DECODE_WARPS, S4KV_DECODE_MIN_CTAS) mq_kernel(DecodeArgs a) {
  using F = Rec<BITS>;
  constexpr int RS = kRecStrideB<BITS>;
  constexpr int kWarps = S4KV_DECODE_WARPS;
  constexpr int kThreads = 32 * kWarps;
  using SmemT = Smem<kWarps>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmemT& sm = *reinterpret_cast<SmemT*>(smem_raw);
  long long* pre = reinterpret_cast<long long*>(smem_raw + prefix_offset<0>());   // [B + 1]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tw = a.tw, tpc = kWarps / tw;
  const int team = warp / tw, tile = warp - team * tw;
  const bool in_team = team < tpc;
  const int lead = in_team ? team * tw : warp;
  const bool leader = in_team && tile == 0;
  uint8_t* st0 = sm.region[lead];
  uint8_t* st1 = st0 + kStageBytesB<BITS>;
  uint64_t* full = sm.bar[lead];
  uint64_t* empty = sm.bar[lead] + kStages;
  float* ptile = sm.ptile[warp];
  // mma_to_gen scratch: a warp's own region (the leader's only once its team is done with it)
  float* scratch = reinterpret_cast<float*>(sm.region[warp]);

  if (leader && lane == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(&empty[0], tw);
    mbar_init(&empty[1], tw);
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __shared__ __align__(16) uint4 zero16;
  if (tid == 0) zero16 = make_uint4(0u, 0u, 0u, 0u);
  const uint32_t zero_s = smem_u32(&zero16);
  {
    long long carry = 0;
    __shared__ long long wt[kWarps];
    for (int base = 0; base < a.B; base += kThreads) {
      const int b = base + tid;
      const long long cnt = b < a.B ? a.H * seg_cost(a.seq_lens[b], a.R, a.tail_cost).cost : 0;
      long long x = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) wt[warp] = x;
      __syncthreads();
      long long before = carry, total = 0;
      for (int q = 0; q < kWarps; ++q) {
        if (q < warp) before += wt[q];
        total += wt[q];
      }
      if (b < a.B) pre[b] = before + x - cnt;
      __syncthreads();
      carry += total;
    }
    if (tid == 0) pre[a.B] = carry;
    __syncthreads();
  }
  const long long C = pre[a.B];
  int n_act = static_cast<int>(gridDim.x) * tpc;
  if (a.max_warps > 0 && a.max_warps < n_act) n_act = a.max_warps;   // the option caps teams here
  {
    const long long cap = (C + kMinUnits - 1) / kMinUnits;
    if (cap < n_act) n_act = static_cast<int>(cap);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!in_team) return;
  const int gteam = blockIdx.x * tpc + team;
  if (gteam >= n_act) return;
  const int gw = blockIdx.x * kWarps + warp;
  const long long r0 = gteam * C / n_act, r1 = (gteam + 1) * C / n_act;
  const uint64_t once = policy_evict_first();
  const int cols = a.nq * a.g;

  uint32_t fph = 0, eph = 0, epend = 0, pend = 0;
  bool aborted = false;
  auto wait_full = [&](int s) -> bool {
    if (!mbar_wait(&full[s], (fph >> s) & 1u, aborted ? 0 : a.wait_ns)) return false;
    fph ^= 1u << s;
    pend &= ~(1u << s);
    return true;
  };
  auto release = [&](int s) {   // this warp is done reading stage s
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&empty[s])) : "memory");
    epend |= 1u << s;
  };
  auto claim = [&](int s) -> bool {   // leader: every warp of the team is done with stage s
    if (!((epend >> s) & 1u)) return true;
    if (!mbar_wait(&empty[s], (eph >> s) & 1u, aborted ? 0 : a.wait_ns)) return false;
    eph ^= 1u << s;
    epend &= ~(1u << s);
    return true;
  };
  auto fail = [&](long long where) {
    if (lane == 0) report(a.status, S4KV_ERR_DEVICE_TIMEOUT, S4KV_DEV_TIMEOUT, static_cast<int>(where));
    aborted = true;
    for (int s = 0; s < kStages; ++s) {
      if ((pend >> s) & 1u) {
        mbar_wait(&full[s], (fph >> s) & 1u, kDrainNs);
        fph ^= 1u << s;
        pend &= ~(1u << s);
      }
    }
  };

  int b;
  {
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  SegCost sc = seg_cost(a.seq_lens[b], a.R, a.tail_cost);
  int h = static_cast<int>((r0 - pre[b]) / sc.cost);
  long long seg_start = pre[b] + h * sc.cost;

  while (seg_start < r1) {
    const long long seg_end = seg_start + sc.cost;
    const int T = max(a.seq_lens[b], 0);
    const long long lo = max(r0, seg_start) - seg_start, hi = min(r1, seg_end) - seg_start;
    const bool own = lo == 0 && hi == sc.cost;
    const int nm = sc.main_groups;
    const int u0 = static_cast<int>(lo < nm ? lo : nm), u1 = static_cast<int>(hi < nm ? hi : nm);
    int c0 = 0, c1 = 0;
    if (sc.tail_chunks > 0 && hi > nm) {
      c0 = static_cast<int>(lo > nm ? (lo - nm + a.tail_cost - 1) / a.tail_cost : 0);
      const long long cc = (hi - nm + a.tail_cost - 1) / a.tail_cost;
      c1 = static_cast<int>(cc < sc.tail_chunks ? cc : sc.tail_chunks);
    }
    const int slot = a.slot_ids ? a.slot_ids[b] : b;
    const bool slot_ok = slot >= 0 && slot < a.max_slots;
    const bool table_ok = static_cast<long long>(a.bt_stride) * kP >= T;
    const int lens_v = slot_ok ? a.lens[slot * a.H + h] : 0;
    Seg sg;
    sg.pages = a.pages;
    sg.bt = a.block_table + static_cast<long long>(b) * a.bt_stride;
    sg.kring = reinterpret_cast<const uint16_t*>(a.kring) + (slot_ok ? slot : 0) * a.kring_slot + h * a.kring_head;
    sg.vring = reinterpret_cast<const uint16_t*>(a.vring) + (slot_ok ? slot : 0) * a.vring_slot + h * a.vring_head;
    sg.H = a.H;
    sg.h = h;
    sg.T = T;
    sg.Tk = T & ~(kG - 1);
    sg.Tv = max(0, T - a.R);
    sg.R = a.R;
    sg.dtype = a.dtype;
    bool valid = slot_ok && T > 0;
    bool bad = false;
    if (valid && table_ok && (u1 > u0 || c1 > c0)) {
      const int p_lo = u1 > u0 ? 2 * u0 : 2 * (nm + c0);
      const int p_hi = min(c1 > c0 ? 2 * (nm + c1) : 2 * u1, (T + kP - 1) / kP);
      for (int base = p_lo; base < p_hi; base += 32 * 8) {
        int pp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int lp = base + 32 * k + lane;
          pp[k] = lp < p_hi ? sg.bt[lp] : 0;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (base + 32 * k + lane < p_hi && (pp[k] < 0 || pp[k] >= a.num_pages)) {
            bad = true;
            report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp[k]);
          }
        }
      }
    }
    if (!slot_ok) {
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
    } else if (lens_v != T || T > a.max_seq_len || T < a.nq) {
      valid = false;
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, b);
    } else if (!table_ok) {
      valid = false;
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, b);
    }
    valid = valid && !__any_sync(0xffffffffu, bad) && !aborted;
    // row of out / q for column c of this segment
    auto row_of = [&](int c) -> long long {
      return (static_cast<long long>(b) * a.nq + c / a.g) * a.Hq + h * a.g + c % a.g;
    };
    GenState gs;
    if (valid) {
      const int n = u1 - u0;
      const int gi = lane >> 2, ti = lane & 3;
      float qv[32];
      {
        const int c = 8 * tile + gi;
        uint4 qraw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) qraw[i] = make_uint4(0u, 0u, 0u, 0u);
        if (c < cols) {
          const uint4* src = reinterpret_cast<const uint4*>(a.q + row_of(c) * kD + 32 * ti);
#pragma unroll
          for (int i = 0; i < 4; ++i) qraw[i] = src[i];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t w[4] = {qraw[i].x, qraw[i].y, qraw[i].z, qraw[i].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            qv[8 * i + 2 * j] = widen16(static_cast<uint16_t>(w[j] & 0xffff), a.dtype);
            qv[8 * i + 2 * j + 1] = widen16(static_cast<uint16_t>(w[j] >> 16), a.dtype);
          }
        }
      }
      // causal limits of this lane's accumulator columns 2ti, 2ti+1 of the tile
      const int ca = 8 * tile + 2 * ti, cb = ca + 1;
      const int lim0 = ca < cols ? T - a.nq + ca / a.g + 1 : T;
      const int lim1 = cb < cols ? T - a.nq + cb / a.g + 1 : T;
      MmaState ms;
      mma_init(ms);
      // leader: pool pages of main groups u0 + 32 k + lane, a batch ahead
      int cur0 = 0, cur1 = 0, nxt0 = 0, nxt1 = 0, cur_k = 0;
      auto load_batch = [&](int k, int& x0, int& x1) {
        const int jj = u0 + 32 * k + lane;
        x0 = x1 = 0;
        if (jj < u1) {
          x0 = sg.bt[2 * jj];
          x1 = sg.bt[2 * jj + 1];
        }
      };
      auto issue_group = [&](int s, int j) {
        if ((j >> 5) != cur_k) {
          cur0 = nxt0;
          cur1 = nxt1;
          ++cur_k;
          load_batch(cur_k + 1, nxt0, nxt1);
        }
        const int p0 = __shfl_sync(0xffffffffu, cur0, j & 31);
        const int p1 = __shfl_sync(0xffffffffu, cur1, j & 31);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          uint8_t* dst = s ? st1 : st0;
          mbar_expect_tx(&full[s], 2 * F::kBytes);
          bulk_load_hint(dst, rec_at<BITS>(sg, p0), F::kBytes, &full[s], once);
          bulk_load_hint(dst + RS, rec_at<BITS>(sg, p1), F::kBytes, &full[s], once);
        }
        pend |= 1u << s;
      };
      bool ok = true;
      if (leader) {
        load_batch(0, cur0, cur1);
        load_batch(1, nxt0, nxt1);
        for (int j = 0; j < n && j < kStages; ++j) {
          if (!claim(j)) { ok = false; break; }
          issue_group(j, j);
        }
      }
      for (int j = 0; ok && j < n; ++j) {
        const int s = j & 1;
        if (!wait_full(s)) { ok = false; break; }
        mma_group<true, BITS>(reinterpret_cast<const char*>(s ? st1 : st0), ms, ptile, qv, a.sm_scale_log2,
                              kLoAbove / a.sm_scale_log2);
        release(s);
        if (leader && j + kStages < n) {
          if (!claim(s)) { ok = false; break; }
          issue_group(s, j + kStages);
        }
      }
      mma_unscale<BITS>(ms);
      int tpg = 0;
      {
        const int lp = 2 * (nm + c0) + lane;
        if (c1 > c0 && lp < min(2 * (nm + c1), (T + kP - 1) / kP)) tpg = sg.bt[lp];
      }
      for (int c = c0; ok && c < c1; ++c) {
        const int grp = nm + c;
        const int t0 = 32 * grp, t1 = min(t0 + kG, T);
        const bool kquant = t0 + kG <= sg.Tk;
        const bool vrec = t0 < sg.Tv;
        const bool kring_staged = !kquant && !vrec && t1 - t0 <= kKringStageMax;
        const int np = (t0 + kP < T) ? 2 : 1;
        const int vt0 = max(t0, sg.Tv);
        const int nv = max(0, t1 - vt0);
        const int voff = kring_staged ? (t1 - t0) * kD * 2 : kVoffRecsB<BITS>;
        const int tp0 = __shfl_sync(0xffffffffu, tpg, (2 * (c - c0)) & 31);
        const int tp1 = __shfl_sync(0xffffffffu, tpg, (2 * (c - c0) + 1) & 31);
        if (leader) {
          // the batch overwrites the whole region: the team must be done with both stages
          if (!claim(0) || !claim(1)) { ok = false; break; }
          uint32_t bytes = nv * kD * 2;
          if (vrec) bytes += np * F::kBytes;
          else if (kquant) bytes += np * (F::kKm + 512);
          if (kring_staged) bytes += (t1 - t0) * kD * 2;
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            mbar_expect_tx(&full[0], bytes);
            if (vrec || kquant) {
              const bool held = c - c0 < 16;
              const char* ra = held ? rec_at<BITS>(sg, tp0) : rec_of<BITS>(sg, 2 * grp);
              const char* rb = np < 2 ? ra : held ? rec_at<BITS>(sg, tp1) : rec_of<BITS>(sg, 2 * grp + 1);
              const uint32_t nb = vrec ? F::kBytes : F::kKm + 512;
              bulk_load_hint(st0, ra, nb, &full[0], once);
              if (np == 2) bulk_load_hint(st0 + RS, rb, nb, &full[0], once);
            }
            if (kring_staged) bulk_load_hint(st0, sg.kring, (t1 - t0) * kD * 2, &full[0], once);
          }
          __syncwarp();
          if (lane < nv) {
            const int t = vt0 + lane;
            bulk_load_hint(st0 + voff + (t - t0) * kVRow, sg.vring + static_cast<long long>(t % sg.R) * kD, kD * 2,
                           &full[0], once);
          }
          pend |= 1u;
        }
        if (!wait_full(0)) { ok = false; break; }
        tail_group<BITS>(sg, grp, ms, ptile, qv, reinterpret_cast<const char*>(st0),
                   kring_staged ? reinterpret_cast<const uint16_t*>(st0) : sg.kring,
                   reinterpret_cast<const char*>(st0 + voff), zero_s, a.sm_scale_log2, lim0, lim1, nullptr);
        release(0);
      }
      if (ok && leader && (!claim(0) || !claim(1))) ok = false;   // scratch below is the staging region
      if (ok) mma_to_gen(ms, gs, scratch);
      else {
        fail(b);
        gen_init(gs);
      }
    } else {
      gen_init(gs);
    }

    // ---- output, or the partial that mq_merge_kernel combines ----
    if (leader && seg_start >= r0 && lane == 0) {
      int ncon = 0;
      if (!own && slot_ok) ncon = owner_of(seg_end - 1, C, n_act) - gteam + 1;
      const long long first = 2LL * gteam + (seg_start <= r0 ? 0 : 1);
      meta_of(a)[static_cast<long long>(b) * a.H + h] =
          static_cast<long long>(static_cast<unsigned>(first)) | (static_cast<long long>(ncon) << 32);
    }
    if (own || !slot_ok) {
#pragma unroll
      for (int j = 0; j < kNH; ++j) {
        const int c = 8 * tile + j;
        if (c < cols) {
          const float inv = gs.l[j] > 0.0f ? 1.0f / gs.l[j] : 0.0f;
          store_out(a, row_of(c), lane,
                    make_float4(gs.o[j][0] * inv, gs.o[j][1] * inv, gs.o[j][2] * inv, gs.o[j][3] * inv));
        }
      }
    } else {
      const int k = seg_start <= r0 ? 0 : 1;
      float* P = a.ws + (2LL * gw + k) * partial_floats(a.pcols);
#pragma unroll
      for (int j = 0; j < kNH; ++j) {
        *reinterpret_cast<float4*>(P + j * kD + 4 * lane) = make_float4(gs.o[j][0], gs.o[j][1], gs.o[j][2], gs.o[j][3]);
        if (lane == 0) {
          P[a.pcols * kD + 2 * j] = gs.m[j];
          P[a.pcols * kD + 2 * j + 1] = gs.l[j];
        }
      }
    }
    seg_start = seg_end;
    if (++h == a.H) {
      h = 0;
      if (++b >= a.B) break;
      sc = seg_cost(a.seq_lens[b], a.R, a.tail_cost);
    }
  }
  if (pend) fail(-1);
}

// Multi-query attention over FP8 pages: the same causal reading and cost line as
// mq_kernel (FP8 segments have no tail), with 16 columns per warp. A team of
// tw = ceil(nq g / 16) warps shares each page record: its leader stages single
// pages into a ring of 2 tw stages spread over the team's regions (full
// barriers), every warp runs fp8_page_mq on its 16 columns and then marks the
// stage free (empty barriers). Partials hold 16 columns (pcols = 16).
__global__ void __launch_bounds__(32 * S4KV_DECODE_WARPS, S4KV_DECODE_MIN_CTAS) mq_fp8_kernel(DecodeArgs a) {
  constexpr int kWarps = S4KV_DECODE_WARPS;
  constexpr int kThreads = 32 * kWarps;
  constexpr int RB = Rec<8>::kBytes;
  static_assert(2 * RB <= kRegion, "two FP8 stages fit a warp's region");
  using SmemT = Smem<kWarps>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmemT& sm = *reinterpret_cast<SmemT*>(smem_raw);
  long long* pre = reinterpret_cast<long long*>(smem_raw + prefix_offset<0>());   // [B + 1]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tw = a.tw, tpc = kWarps / tw;
  const int team = warp / tw, tile = warp - team * tw;
  const bool in_team = team < tpc;
  const int lead = in_team ? team * tw : warp;
  const bool leader = in_team && tile == 0;
  const int NS = 2 * tw;   // stage s: region of warp lead + s / 2, half s % 2
  auto stage = [&](int s) -> uint8_t* { return sm.region[lead + (s >> 1)] + (s & 1) * RB; };
  auto full_of = [&](int s) -> uint64_t* { return &sm.bar[lead + (s >> 1)][s & 1]; };
  auto empty_of = [&](int s) -> uint64_t* { return &sm.bar[lead + (s >> 1)][kStages + (s & 1)]; };
  float* scratch = reinterpret_cast<float*>(sm.region[warp]);   // mma_to_gen, once the team is done

  if (in_team && lane == 0) {
    mbar_init(&sm.bar[warp][0], 1);
    mbar_init(&sm.bar[warp][1], 1);
    mbar_init(&sm.bar[warp][kStages], tw);
    mbar_init(&sm.bar[warp][kStages + 1], tw);
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  {
    long long carry = 0;
    __shared__ long long wt[kWarps];
    for (int base = 0; base < a.B; base += kThreads) {
      const int b = base + tid;
      const long long cnt = b < a.B ? a.H * seg_cost<8>(a.seq_lens[b], a.R, a.tail_cost).cost : 0;
      long long x = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) wt[warp] = x;
      __syncthreads();
      long long before = carry, total = 0;
      for (int q = 0; q < kWarps; ++q) {
        if (q < warp) before += wt[q];
        total += wt[q];
      }
      if (b < a.B) pre[b] = before + x - cnt;
      __syncthreads();
      carry += total;
    }
    if (tid == 0) pre[a.B] = carry;
    __syncthreads();
  }
  const long long C = pre[a.B];
  int n_act = static_cast<int>(gridDim.x) * tpc;
  if (a.max_warps > 0 && a.max_warps < n_act) n_act = a.max_warps;   // the option caps teams here
  {
    const long long cap = (C + kMinUnits - 1) / kMinUnits;
    if (cap < n_act) n_act = static_cast<int>(cap);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!in_team) return;
  const int gteam = blockIdx.x * tpc + team;
  if (gteam >= n_act) return;
  const int gw = blockIdx.x * kWarps + warp;
  const long long r0 = gteam * C / n_act, r1 = (gteam + 1) * C / n_act;
  const uint64_t once = policy_evict_first();
  const int cols = a.nq * a.g;
  const int gi = lane >> 2, ti = lane & 3;
  auto team_sync = [&]() {   // named barrier of the team's warps (id 0 is __syncthreads)
    if (tw > 1) asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(32 * tw) : "memory");
    else __syncwarp();
  };

  uint32_t fph = 0, eph = 0, epend = 0, pend = 0;
  bool aborted = false;
  auto wait_full = [&](int s) -> bool {
    if (!mbar_wait(full_of(s), (fph >> s) & 1u, aborted ? 0 : a.wait_ns)) return false;
    fph ^= 1u << s;
    pend &= ~(1u << s);
    return true;
  };
  auto release = [&](int s) {   // this warp is done reading stage s
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(empty_of(s))) : "memory");
    epend |= 1u << s;
  };
  auto claim = [&](int s) -> bool {   // leader: every warp of the team is done with stage s
    if (!((epend >> s) & 1u)) return true;
    if (!mbar_wait(empty_of(s), (eph >> s) & 1u, aborted ? 0 : a.wait_ns)) return false;
    eph ^= 1u << s;
    epend &= ~(1u << s);
    return true;
  };
  auto fail = [&](long long where) {
    if (lane == 0) report(a.status, S4KV_ERR_DEVICE_TIMEOUT, S4KV_DEV_TIMEOUT, static_cast<int>(where));
    aborted = true;
    for (int s = 0; s < NS; ++s) {
      if ((pend >> s) & 1u) {
        mbar_wait(full_of(s), (fph >> s) & 1u, kDrainNs);
        fph ^= 1u << s;
        pend &= ~(1u << s);
      }
    }
  };

  int b;
  {
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  SegCost sc = seg_cost<8>(a.seq_lens[b], a.R, a.tail_cost);
  int h = static_cast<int>((r0 - pre[b]) / sc.cost);
  long long seg_start = pre[b] + h * sc.cost;

  while (seg_start < r1) {
    const long long seg_end = seg_start + sc.cost;
    const int T = max(a.seq_lens[b], 0);
    const long long lo = max(r0, seg_start) - seg_start, hi = min(r1, seg_end) - seg_start;
    const bool own = lo == 0 && hi == sc.cost;
    const int nm = sc.main_groups;
    const int u0 = static_cast<int>(lo < nm ? lo : nm), u1 = static_cast<int>(hi < nm ? hi : nm);
    const int slot = a.slot_ids ? a.slot_ids[b] : b;
    const bool slot_ok = slot >= 0 && slot < a.max_slots;
    const bool table_ok = static_cast<long long>(a.bt_stride) * kP >= T;
    const int lens_v = slot_ok ? a.lens[slot * a.H + h] : 0;
    const float ks = a.fp8_scale[h], vs = a.fp8_scale[a.H + h];
    Seg sg;
    sg.pages = a.pages;
    sg.bt = a.block_table + static_cast<long long>(b) * a.bt_stride;
    sg.H = a.H;
    sg.h = h;
    sg.T = T;
    const int npT = (T + kP - 1) / kP;
    const int pg0 = 2 * u0, pg1 = min(2 * u1, npT), np = max(0, pg1 - pg0);
    bool valid = slot_ok && T > 0;
    bool bad = false;
    if (valid && table_ok && np > 0) {
      for (int base = pg0; base < pg1; base += 32 * 8) {
        int pp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int lp = base + 32 * k + lane;
          pp[k] = lp < pg1 ? sg.bt[lp] : 0;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (base + 32 * k + lane < pg1 && (pp[k] < 0 || pp[k] >= a.num_pages)) {
            bad = true;
            report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp[k]);
          }
        }
      }
    }
    if (!slot_ok) {
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
    } else if (lens_v != T || T > a.max_seq_len || T < a.nq) {
      valid = false;
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, b);
    } else if (!table_ok) {
      valid = false;
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, b);
    }
    valid = valid && !__any_sync(0xffffffffu, bad) && !aborted;
    auto row_of = [&](int c) -> long long {
      return (static_cast<long long>(b) * a.nq + c / a.g) * a.Hq + h * a.g + c % a.g;
    };
    float o[8][2][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int ct = 0; ct < 2; ++ct)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][ct][e] = 0.0f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
    bool ok = true;
    if (valid) {
      // A operand rows: columns c_lo = 16 tile + gi and c_hi = c_lo + 8 (zero past cols)
      const int c_lo = 16 * tile + gi, c_hi = c_lo + 8;
      uint32_t qa[8][4];
      {
        uint4 ql[4], qh[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ql[i] = qh[i] = make_uint4(0u, 0u, 0u, 0u);
        if (c_lo < cols) {
          const uint4* src = reinterpret_cast<const uint4*>(a.q + row_of(c_lo) * kD + 32 * ti);
#pragma unroll
          for (int i = 0; i < 4; ++i) ql[i] = src[i];
        }
        if (c_hi < cols) {
          const uint4* src = reinterpret_cast<const uint4*>(a.q + row_of(c_hi) * kD + 32 * ti);
#pragma unroll
          for (int i = 0; i < 4; ++i) qh[i] = src[i];
        }
        // channel 32 ti + 4 kk + j sits in word (kk / 2) of uint4 i = kk / 2 ... as 16-bit halves:
        // q words hold channels 32 ti + 2 w, + 1 (w = 0 .. 15)
        auto q2 = [&](const uint4 (&u)[4], int w) -> uint32_t {   // channels 32 ti + 2w, 2w + 1 as f16x2
          const uint4 x = u[w >> 2];
          const uint32_t r = (w & 3) == 0 ? x.x : (w & 3) == 1 ? x.y : (w & 3) == 2 ? x.z : x.w;
          if (a.dtype == S4KV_F16) return r;
          return pack_f16x2(widen16(static_cast<uint16_t>(r & 0xffff), S4KV_BF16),
                            widen16(static_cast<uint16_t>(r >> 16), S4KV_BF16));
        };
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          qa[kk][0] = q2(ql, 2 * kk);       // column c_lo, channels c_0, c_1
          qa[kk][1] = q2(qh, 2 * kk);       // column c_hi, c_0, c_1
          qa[kk][2] = q2(ql, 2 * kk + 1);   // column c_lo, c_2, c_3
          qa[kk][3] = q2(qh, 2 * kk + 1);
        }
      }
      // causal limits; pages wholly below every column's limit need no mask
      const int lim_lo = c_lo < cols ? T - a.nq + c_lo / a.g + 1 : T;
      const int lim_hi = c_hi < cols ? T - a.nq + c_hi / a.g + 1 : T;
      int free_end = min(lim_lo, lim_hi);
#pragma unroll
      for (int x = 1; x < 32; x <<= 1) free_end = min(free_end, __shfl_xor_sync(0xffffffffu, free_end, x));
      const float zscale = a.sm_scale_log2 * ks;
      // leader: pool pages pg0 + 32 k + lane, one batch of 32 ahead of the copies
      auto page_of = [&](int k) {
        const int lp = pg0 + 32 * k + lane;
        return lp < pg1 ? sg.bt[lp] : 0;
      };
      int curp = 0, nxtp = 0, cur_k = 0;
      auto issue_page = [&](int s, int i) {   // i = 0, 1, 2, ... in order
        if ((i >> 5) != cur_k) {
          curp = nxtp;
          ++cur_k;
          nxtp = page_of(cur_k + 1);
        }
        const int pp = __shfl_sync(0xffffffffu, curp, i & 31);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          mbar_expect_tx(full_of(s), RB);
          bulk_load_hint(stage(s), rec_at<8>(sg, pp), RB, full_of(s), once);
        }
        pend |= 1u << s;
      };
      if (leader) {
        curp = page_of(0);
        nxtp = page_of(1);
        for (int i = 0; i < np && i < NS; ++i) {
          if (!claim(i)) { ok = false; break; }
          issue_page(i, i);
        }
      }
      for (int i = 0, s = 0; ok && i < np; ++i) {
        if (!wait_full(s)) { ok = false; break; }
        const char* rec = reinterpret_cast<const char*>(stage(s));
        const int tok0 = kP * (pg0 + i);
        if (tok0 + kP > free_end) fp8_page_mq<true>(rec, o, m, l, qa, zscale, tok0, lim_lo, lim_hi, T - tok0);
        else fp8_page_mq<false>(rec, o, m, l, qa, zscale, tok0, lim_lo, lim_hi, kP);
        release(s);
        if (leader && i + NS < np) {
          if (!claim(s)) { ok = false; break; }
          issue_page(s, i + NS);
        }
        s = s + 1 == NS ? 0 : s + 1;
      }
      if (!ok) {
        fail(b);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int ct = 0; ct < 2; ++ct)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][ct][e] = 0.0f;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.0f;
      }
    }
    // every warp of the team is done reading the stages in its region before it
    // writes its scratch there (each warp passes these barriers once per segment)
    team_sync();
    // sums of columns gi, gi + 8 over the lane's four token positions
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
      l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
    }
    if (leader && seg_start >= r0 && lane == 0) {
      int ncon = 0;
      if (!own && slot_ok) ncon = owner_of(seg_end - 1, C, n_act) - gteam + 1;
      const long long first = 2LL * gteam + (seg_start <= r0 ? 0 : 1);
      meta_of(a)[static_cast<long long>(b) * a.H + h] =
          static_cast<long long>(static_cast<unsigned>(first)) | (static_cast<long long>(ncon) << 32);
    }
#pragma unroll
    for (int ct = 0; ct < 2; ++ct) {
      // column tile ct (columns 16 tile + 8 ct + j) in the two-columns-per-lane form of mma_to_gen
      MmaState ms;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) ms.o[mt][e] = o[mt][ct][e] * vs;
#pragma unroll
      for (int k = 0; k < 4; ++k) ms.bias[k] = 0.0f;
      ms.m0 = __shfl_sync(0xffffffffu, m[ct], 8 * ti);
      ms.m1 = __shfl_sync(0xffffffffu, m[ct], 8 * ti + 4);
      const float lt0 = __shfl_sync(0xffffffffu, l[ct], 8 * ti), lt1 = __shfl_sync(0xffffffffu, l[ct], 8 * ti + 4);
      ms.l0 = lane < 4 ? lt0 : 0.0f;
      ms.l1 = lane < 4 ? lt1 : 0.0f;
      GenState gs;
      mma_to_gen(ms, gs, scratch);
      if (own || !slot_ok) {
#pragma unroll
        for (int j = 0; j < kNH; ++j) {
          const int c = 16 * tile + 8 * ct + j;
          if (c < cols) {
            const float inv = gs.l[j] > 0.0f ? 1.0f / gs.l[j] : 0.0f;
            store_out(a, row_of(c), lane,
                      make_float4(gs.o[j][0] * inv, gs.o[j][1] * inv, gs.o[j][2] * inv, gs.o[j][3] * inv));
          }
        }
      } else {
        const int k = seg_start <= r0 ? 0 : 1;
        float* P = a.ws + (2LL * gw + k) * partial_floats(a.pcols);
#pragma unroll
        for (int j = 0; j < kNH; ++j) {
          const int jj = 8 * ct + j;
          *reinterpret_cast<float4*>(P + jj * kD + 4 * lane) =
              make_float4(gs.o[j][0], gs.o[j][1], gs.o[j][2], gs.o[j][3]);
          if (lane == 0) {
            P[a.pcols * kD + 2 * jj] = gs.m[j];
            P[a.pcols * kD + 2 * jj + 1] = gs.l[j];
          }
        }
      }
    }
    fence_proxy_async();   // the scratch writes come before later bulk copies into the region
    team_sync();
    seg_start = seg_end;
    if (++h == a.H) {
      h = 0;
      if (++b >= a.B) break;
      sc = seg_cost<8>(a.seq_lens[b], a.R, a.tail_cost);
    }
  }
  if (pend) fail(-1);
}

// ---- multi-query over KIVI pages: each key group restored once to shared memory ----------
// A team restores each 32-token group once for all its columns: K^ = code * scale
// + min in fp32 (as the restore defines it), kept as an f16 high part plus the f16
// rest (about 22 bits; a key scale folded into the query in f16 would be the
// larger error on wide-scale channels), and V^ in f16. Keys past the quantized
// range come from the key ring (split the same way), values past it from the
// value ring, and tokens past T are zero. Each warp then runs plain MMAs from
// shared memory on its 16 (query, head) columns: the columns are the rows of the
// key-score MMA and the probabilities feed P V from registers, as for FP8 pages.
constexpr int kKRow = 2 * kD + 16;   // K^ rows, token-major: 272 B (ldmatrix rows in distinct banks)
constexpr int kVTRow = 2 * kG + 16;  // V^T rows, channel-major over a group's 32 tokens: 80 B
template <int BITS>
struct MqSmem {                      // byte offsets in a team's block of warp regions
  static constexpr int kStage = kStageBytesB<BITS>;   // two page records
  static constexpr int kKhi = 2 * kStage;
  static constexpr int kKlo = kKhi + kG * kKRow;
  static constexpr int kVt = kKlo + kG * kKRow;
  static constexpr int kEnd = kVt + kD * kVTRow;
};
constexpr int kMqMinTeam = (MqSmem<4>::kEnd + kRegion - 1) / kRegion;   // warps whose regions hold it
static_assert(MqSmem<4>::kStage % 16 == 0 && MqSmem<2>::kStage % 16 == 0 && MqSmem<4>::kEnd >= MqSmem<2>::kEnd,
              "16-byte aligned stages; 4-bit records take the most room");
static_assert(kMqMinTeam * 2 <= S4KV_DECODE_WARPS, "at least two restoring teams per CTA");

// byte of a key or value word that holds channel c_j (keys) / column j
__device__ __forceinline__ int byte_of_j(int j) { return j == 1 ? 2 : j == 2 ? 1 : j; }

// A code (0 .. 255) as a float, exactly: 2^23 + n holds n in its low mantissa bits.
__device__ __forceinline__ float code_f(uint32_t n) { return __fsub_rn(__uint_as_float(0x4B000000u | n), 8388608.0f); }

// Veltkamp split of x: hi keeps the top 11 significant bits (exact in f16 within
// its range), lo = x - hi exactly; lo rounded to f16 leaves about 22 bits in all.
__device__ __forceinline__ void split11(float x, float& hi, float& lo) {
  const float c = __fmul_rn(x, 8193.0f);   // 2^13 + 1
  hi = __fsub_rn(c, __fsub_rn(c, x));
  lo = __fsub_rn(x, hi);
}

__device__ __forceinline__ void store_hi_lo(char* hi_row, char* lo_row, const float (&x)[8]) {
  uint32_t h[4], r[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    float h0, l0, h1, l1;
    split11(x[2 * p], h0, l0);
    split11(x[2 * p + 1], h1, l1);
    h[p] = pack_f16x2(h0, h1);
    r[p] = pack_f16x2(l0, l1);
  }
  *reinterpret_cast<uint4*>(hi_row) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo_row) = make_uint4(r[0], r[1], r[2], r[3]);
}

// Byte offset of element (row r, column k) of a K-major tcgen05 operand in the
// no-swizzle core-matrix layout: 8-row x 16-byte core matrices, the next one along
// K 128 bytes on (LBO), the next 8 rows `sbo` bytes on (SBO).
__device__ __forceinline__ int core_off(int r, int k, int sbo) {
  return (r >> 3) * sbo + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}
constexpr int kCoreSbo128 = 16 * 128;   // operands with K = 128 (channels)
constexpr int kCoreSbo32 = 4 * 128;     // operands with K = 32 (a group's tokens)

// ---- tcgen05: 5th-generation tensor cores, accumulators in tensor memory -------------------
// Shared-memory operand descriptor of a K-major operand in the no-swizzle core-matrix
// layout (core_off): start address / 16, leading byte offset 128 / 16 (the next core
// matrix along K), stride byte offset / 16 (the next 8 rows), descriptor version 1.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(128 >> 4) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46);
}
// Instruction descriptor of kind::f16: f32 accumulator, f16 A and B, both K-major, N / 8, M / 16.
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
// D[tmem] (+)= A B^T, one thread issues; acc = false overwrites D.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc ? 1u : 0u)
      : "memory");
}
// `bar` receives one arrival once the MMAs this thread issued so far have completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 32 consecutive 32-bit columns of this thread's TMEM lane (warp w addresses lanes 32 (w % 4) ..).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]) : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Keys of group tokens t0 .. t0 + 31: thread thr of nthr takes (token, 8 channels)
// items. kTail: a token may be past the quantized keys (ring) or past T (zero).
// kCore: K^ in the core-matrix layout (rows = tokens, K = channels), else rows of kKRow.
template <int BITS, bool kTail, bool kCore = false>
__device__ void restore_keys(const char* stage, char* khi, char* klo, int t0, int T, int Tk,
                             const uint16_t* kring, int dtype, int thr, int nthr) {
  using F = Rec<BITS>;
  constexpr int RS = kRecStrideB<BITS>;
  for (int it = thr; it < kG * 16; it += nthr) {
    // core layout: consecutive threads take consecutive tokens (conflict-free stores)
    const int tau = kCore ? (it & 31) : (it >> 4), c0 = 8 * (kCore ? (it >> 5) : (it & 15));
    const int t = t0 + tau;
    float x[8];
    if (!kTail || t < Tk) {
      // channel 32 b + 4 kk + j: slices kk0 (j = 0..3 of c0..c0+3) and kk0 + 1 (c0+4..c0+7)
      const char* rec = stage + (tau >> 4) * RS;
      const int tp = tau & 15, hi = tp >> 3, L = 4 * (tp & 7) + (c0 >> 5), kk0 = (c0 & 31) >> 2;
      uint32_t code[8];
      if constexpr (BITS == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(rec + F::kKc + (kk0 >> 2) * 512 + L * 16 + (kk0 & 3) * 4);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          code[j] = (w.x >> (8 * byte_of_j(j) + 4 * hi)) & 15;
          code[4 + j] = (w.y >> (8 * byte_of_j(j) + 4 * hi)) & 15;
        }
      } else {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(rec + F::kKc + L * 16 + (kk0 >> 1) * 4);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          code[j] = (w >> (8 * byte_of_j(j) + 2 * hi)) & 3;
          code[4 + j] = (w >> (8 * byte_of_j(j) + 2 * (2 + hi))) & 3;
        }
      }
      // scale / min of channels c0 .. c0 + 7 in the group's page of channel half c0 / 64
      const char* mrec = stage + (c0 >> 6) * RS + F::kKm;
      const int cl = c0 & 63, u = cl >> 5, i0 = (cl & 31) >> 2;
      const float4 sa = *reinterpret_cast<const float4*>(mrec + (2 * i0 + u) * 16);
      const float4 sb = *reinterpret_cast<const float4*>(mrec + (2 * i0 + 2 + u) * 16);
      const float4 ma = *reinterpret_cast<const float4*>(mrec + 256 + (2 * i0 + u) * 16);
      const float4 mb = *reinterpret_cast<const float4*>(mrec + 256 + (2 * i0 + 2 + u) * 16);
      const float s[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
      const float mn[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = fmaf(code_f(code[j]), s[j], mn[j]);
    } else if (t < T) {
      const uint4 r = *reinterpret_cast<const uint4*>(kring + static_cast<long long>(t % kG) * kD + c0);
      const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        x[2 * p] = widen16(static_cast<uint16_t>(rw[p] & 0xffff), dtype);
        x[2 * p + 1] = widen16(static_cast<uint16_t>(rw[p] >> 16), dtype);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = 0.0f;
    }
    const int off = kCore ? core_off(tau, c0, kCoreSbo128) : tau * kKRow + 2 * c0;
    store_hi_lo(khi + off, klo + off, x);
  }
}

// Values of the group into V^T (channel-major): thread thr of nthr takes code
// words (a word holds 4 tokens of 2 channels at 4 bits, of 4 channels at 2 bits).
// kTail: a token may be past the quantized values (ring) or past T (zero).
// kCore: V^ (rows = channels, K = the group's tokens) in the core-matrix layout.
template <int BITS, bool kTail, bool kCore = false>
__device__ void restore_values(const char* stage, char* vt, int t0, int T, int Tv, const uint16_t* vring, int R,
                               int dtype, int thr, int nthr) {
  using F = Rec<BITS>;
  constexpr int RS = kRecStrideB<BITS>;
  constexpr int kWords = (BITS == 4 ? 8 : 4) * 32;   // per page
  constexpr int kCh = BITS == 4 ? 2 : 4;             // channels per byte
  for (int it = thr; it < 2 * kWords; it += nthr) {
    const int p = it / kWords, wi = it % kWords;
    const int L = wi & 31, mw = wi >> 5;              // word (mt or mp, L)
    const int a = L >> 2, b = L & 3;
    const int tb = t0 + 16 * p;                       // first token of the page
    const char* rec = stage + p * RS;
    // byte i of the word holds page token tok[i]; e[i]: its entry in the metadata quad
    const int tok[4] = {2 * b, 2 * b + 8, 2 * b + 1, 2 * b + 9};
    const int e[4] = {0, 2, 1, 3};
    const bool quant = !kTail || tb < Tv;             // any token of the page quantized
    uint32_t w = 0;
    float4 s4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), m4 = s4;
    if (quant) {
      const int k = BITS == 4 ? (mw >> 1) : mw;       // value group of the word's channels
      w = BITS == 4 ? *reinterpret_cast<const uint32_t*>(rec + F::kVc + (mw >> 2) * 512 + L * 16 + (mw & 3) * 4)
                    : *reinterpret_cast<const uint32_t*>(rec + F::kVc + L * 16 + mw * 4);
      s4 = *reinterpret_cast<const float4*>(rec + F::kVm + ((2 * k) * 4 + b) * 16);
      m4 = *reinterpret_cast<const float4*>(rec + F::kVm + ((2 * k + 1) * 4 + b) * 16);
    }
    const float sq[4] = {s4.x, s4.y, s4.z, s4.w}, mq[4] = {m4.x, m4.y, m4.z, m4.w};
    float v[kCh][4];   // [channel slot][byte]
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = tb + tok[i];
#pragma unroll
      for (int q = 0; q < kCh; ++q) {
        const int ch = BITS == 4 ? 16 * mw + a + 8 * q : 32 * mw + 8 * q + a;
        float x = 0.0f;
        if (!kTail || t < Tv) {
          const uint32_t code = BITS == 4 ? (w >> (8 * i + 4 * q)) & 15u : (w >> (8 * i + 2 * q)) & 3u;
          x = fmaf(code_f(code), sq[e[i]], mq[e[i]]);
        } else if (t < T) {
          x = widen16(vring[static_cast<long long>(t % R) * kD + ch], dtype);
        }
        v[q][i] = x;
      }
    }
#pragma unroll
    for (int q = 0; q < kCh; ++q) {
      const int ch = BITS == 4 ? 16 * mw + a + 8 * q : 32 * mw + 8 * q + a;
      char* row = vt + (kCore ? core_off(ch, 16 * p + 2 * b, kCoreSbo32) : ch * kVTRow + 2 * (16 * p + 2 * b));
      *reinterpret_cast<uint32_t*>(row) = pack_f16x2(v[q][0], v[q][2]);        // tokens 2b, 2b + 1
      // tokens 2b + 8, 2b + 9: the next core matrix along K, or 16 bytes on in a row
      *reinterpret_cast<uint32_t*>(row + (kCore ? 128 : 16)) = pack_f16x2(v[q][1], v[q][3]);
    }
  }
}

// One restored group for a warp's 16 columns (rows gi: column c_lo, gi + 8:
// c_hi): scores from K^ (high and low parts) by MMA, causal mask (kMask: the
// group reaches some column's limit), lazy online softmax, P V from V^T.
template <bool kMask>
__device__ __forceinline__ void mq_group_mma(uint32_t khi, uint32_t klo, uint32_t vt, float (&o)[8][2][4],
                                             float (&m)[2], float (&l)[2], const uint32_t (&qa)[8][4],
                                             float scale, int t0, int lim_lo, int lim_hi) {
  const int lane = threadIdx.x & 31, ti = lane & 3;
  const int j = lane >> 3, r = lane & 7;
  // ldmatrix rows: K^ token 8 (j / 2) + r, channels + 8 (j % 2); V^T channel 8 (j % 2) + r, tokens + 8 (j / 2)
  const uint32_t kofs = (8 * (j >> 1) + r) * kKRow + 16 * (j & 1);
  const uint32_t vofs = (8 * (j & 1) + r) * kVTRow + 16 * (j >> 1);
  float acc[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    uint32_t h0[4], h1[4], l0[4], l1[4];   // tokens 0-15 and 16-31: {b0, b1} of two n8 tiles each
    ldsm_x4(khi + kofs + 32 * kk, h0);
    ldsm_x4(khi + kofs + 16 * kKRow + 32 * kk, h1);
    ldsm_x4(klo + kofs + 32 * kk, l0);
    ldsm_x4(klo + kofs + 16 * kKRow + 32 * kk, l1);
    mma16816(acc[0], qa[kk], h0[0], h0[1]);
    mma16816(acc[1], qa[kk], h0[2], h0[3]);
    mma16816(acc[2], qa[kk], h1[0], h1[1]);
    mma16816(acc[3], qa[kk], h1[2], h1[3]);
    mma16816(acc[0], qa[kk], l0[0], l0[1]);
    mma16816(acc[1], qa[kk], l0[2], l0[3]);
    mma16816(acc[2], qa[kk], l1[0], l1[1]);
    mma16816(acc[3], qa[kk], l1[2], l1[3]);
  }
  // z[row][tile][x]: column row (0: c_lo, 1: c_hi), token t0 + 8 tile + 2 ti + x
  float z[2][4][2];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    z[0][nt][0] = acc[nt][0] * scale;
    z[0][nt][1] = acc[nt][1] * scale;
    z[1][nt][0] = acc[nt][2] * scale;
    z[1][nt][1] = acc[nt][3] * scale;
    if (kMask) {
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int t = t0 + 8 * nt + 2 * ti + x;
        z[0][nt][x] = t < lim_lo ? z[0][nt][x] : -INFINITY;
        z[1][nt][x] = t < lim_hi ? z[1][nt][x] : -INFINITY;
      }
    }
  }
  float mx[2];
#pragma unroll
  for (int rw = 0; rw < 2; ++rw) {
    mx[rw] = z[rw][0][0];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) mx[rw] = fmaxf(mx[rw], fmaxf(z[rw][nt][0], z[rw][nt][1]));
    mx[rw] = fmaxf(mx[rw], __shfl_xor_sync(0xffffffffu, mx[rw], 1));
    mx[rw] = fmaxf(mx[rw], __shfl_xor_sync(0xffffffffu, mx[rw], 2));
  }
  if (__any_sync(0xffffffffu, mx[0] > m[0] + kLazy || mx[1] > m[1] + kLazy)) {
    float al[2];
#pragma unroll
    for (int rw = 0; rw < 2; ++rw) {
      const float mn = fmaxf(m[rw], mx[rw]);
      al[rw] = mn == -INFINITY ? 1.0f : ex2(m[rw] - mn);
      m[rw] = mn;
      l[rw] *= al[rw];
    }
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
  uint32_t pb[2][4][1];   // packed p: [row][tile] (tokens 2ti, 2ti + 1 of the tile)
#pragma unroll
  for (int rw = 0; rw < 2; ++rw) {
    float sum = 0.0f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float p0 = z[rw][nt][0] == -INFINITY ? 0.0f : ex2(z[rw][nt][0] - m[rw]);
      const float p1 = z[rw][nt][1] == -INFINITY ? 0.0f : ex2(z[rw][nt][1] - m[rw]);
      sum += p0 + p1;
      pb[rw][nt][0] = pack_f16x2(p0, p1);
    }
    l[rw] += sum;
  }
#pragma unroll
  for (int pg = 0; pg < 2; ++pg) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t av[4];   // V^T of channels 16 mt .. + 15, tokens 16 pg .. + 15
      ldsm_x4(vt + vofs + 16 * mt * kVTRow + 32 * pg, av);
      mma16816(o[mt][0], av, pb[0][2 * pg][0], pb[0][2 * pg + 1][0]);
      mma16816(o[mt][1], av, pb[1][2 * pg][0], pb[1][2 * pg + 1][0]);
    }
  }
}

// Multi-query attention over KIVI pages (4- or 2-bit), the same causal reading
// and cost line as mq_kernel: teams of tw = max(kMqMinTeam, ceil(nq g / 16)) warps.
// Per key group: the leader's bounded wait on the group's records (its outcome
// shared through shared memory), the team restores the group, the leader stages
// the group two ahead, the column warps run mq_group_mma. Named team barriers
// separate the phases; every warp of a team passes each barrier equally often.
template <int BITS>
__global__ void __launch_bounds__(32 * S4KV_DECODE_WARPS, S4KV_DECODE_MIN_CTAS) mqd_kernel(DecodeArgs a) {
  using F = Rec<BITS>;
  using M = MqSmem<BITS>;
  constexpr int kWarps = S4KV_DECODE_WARPS;
  constexpr int kThreads = 32 * kWarps;
  using SmemT = Smem<kWarps>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmemT& sm = *reinterpret_cast<SmemT*>(smem_raw);
  long long* pre = reinterpret_cast<long long*>(smem_raw + prefix_offset<0>());   // [B + 1]
  __shared__ int team_ok[kWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tw = a.tw, tpc = kWarps / tw;
  const int team = warp / tw, tile = warp - team * tw;
  const bool in_team = team < tpc;
  const int lead = in_team ? team * tw : warp;
  const bool leader = in_team && tile == 0;
  const int cols = a.nq * a.g;
  const int ncw = (cols + 15) / 16;   // warps with columns; the others only restore
  const bool colw = tile < ncw;
  char* blk = reinterpret_cast<char*>(sm.region[lead]);   // the team's regions, contiguous
  float* scratch = reinterpret_cast<float*>(sm.region[warp]);
  uint64_t* full = sm.bar[lead];

  if (leader && lane == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  {
    long long carry = 0;
    __shared__ long long wt[kWarps];
    for (int base = 0; base < a.B; base += kThreads) {
      const int b = base + tid;
      const long long cnt = b < a.B ? a.H * seg_cost(a.seq_lens[b], a.R, a.tail_cost).cost : 0;
      long long x = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) wt[warp] = x;
      __syncthreads();
      long long before = carry, total = 0;
      for (int q = 0; q < kWarps; ++q) {
        if (q < warp) before += wt[q];
        total += wt[q];
      }
      if (b < a.B) pre[b] = before + x - cnt;
      __syncthreads();
      carry += total;
    }
    if (tid == 0) pre[a.B] = carry;
    __syncthreads();
  }
  const long long C = pre[a.B];
  int n_act = static_cast<int>(gridDim.x) * tpc;
  if (a.max_warps > 0 && a.max_warps < n_act) n_act = a.max_warps;   // the option caps teams here
  {
    const long long cap = (C + kMinUnits - 1) / kMinUnits;
    if (cap < n_act) n_act = static_cast<int>(cap);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!in_team) return;
  const int gteam = blockIdx.x * tpc + team;
  if (gteam >= n_act) return;
  const int gw = blockIdx.x * kWarps + warp;
  const long long r0 = gteam * C / n_act, r1 = (gteam + 1) * C / n_act;
  const uint64_t once = policy_evict_first();
  const int gi = lane >> 2, ti = lane & 3;
  const int thr = 32 * tile + lane, nthr = 32 * tw;
  auto team_sync = [&]() {   // named barrier of the team (id 0 is __syncthreads); tw >= 3
    asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(32 * tw) : "memory");
  };
  uint32_t fph = 0, pend = 0;   // leader: stage parities and copies in flight
  bool aborted = false;

  int b;
  {
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  SegCost sc = seg_cost(a.seq_lens[b], a.R, a.tail_cost);
  int h = static_cast<int>((r0 - pre[b]) / sc.cost);
  long long seg_start = pre[b] + h * sc.cost;

  while (seg_start < r1) {
    const long long seg_end = seg_start + sc.cost;
    const int T = max(a.seq_lens[b], 0);
    const long long lo = max(r0, seg_start) - seg_start, hi = min(r1, seg_end) - seg_start;
    const bool own = lo == 0 && hi == sc.cost;
    const int nm = sc.main_groups;
    const int u0 = static_cast<int>(lo < nm ? lo : nm), u1 = static_cast<int>(hi < nm ? hi : nm);
    int c0 = 0, c1 = 0;
    if (sc.tail_chunks > 0 && hi > nm) {
      c0 = static_cast<int>(lo > nm ? (lo - nm + a.tail_cost - 1) / a.tail_cost : 0);
      const long long cc = (hi - nm + a.tail_cost - 1) / a.tail_cost;
      c1 = static_cast<int>(cc < sc.tail_chunks ? cc : sc.tail_chunks);
    }
    const int nmain = u1 - u0, ng = nmain + (c1 - c0);
    auto group_of = [&](int i) { return i < nmain ? u0 + i : nm + c0 + (i - nmain); };
    const int slot = a.slot_ids ? a.slot_ids[b] : b;
    const bool slot_ok = slot >= 0 && slot < a.max_slots;
    const bool table_ok = static_cast<long long>(a.bt_stride) * kP >= T;
    const int lens_v = slot_ok ? a.lens[slot * a.H + h] : 0;
    Seg sg;
    sg.pages = a.pages;
    sg.bt = a.block_table + static_cast<long long>(b) * a.bt_stride;
    sg.H = a.H;
    sg.h = h;
    sg.T = T;
    const int npT = (T + kP - 1) / kP;
    const int Tk = T & ~(kG - 1), Tv = max(0, T - a.R);
    const uint16_t* kring = reinterpret_cast<const uint16_t*>(a.kring) + (slot_ok ? slot : 0) * a.kring_slot + h * a.kring_head;
    const uint16_t* vring = reinterpret_cast<const uint16_t*>(a.vring) + (slot_ok ? slot : 0) * a.vring_slot + h * a.vring_head;
    bool valid = slot_ok && T > 0;
    bool bad = false;
    if (valid && table_ok && ng > 0) {
      const int p_lo = 2 * group_of(0), p_hi = min(2 * group_of(ng - 1) + 2, npT);
      for (int base = p_lo; base < p_hi; base += 32 * 8) {
        int pp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int lp = base + 32 * k + lane;
          pp[k] = lp < p_hi ? sg.bt[lp] : 0;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (base + 32 * k + lane < p_hi && (pp[k] < 0 || pp[k] >= a.num_pages)) {
            bad = true;
            report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp[k]);
          }
        }
      }
    }
    if (!slot_ok) {
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
    } else if (lens_v != T || T > a.max_seq_len || T < a.nq) {
      valid = false;
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, b);
    } else if (!table_ok) {
      valid = false;
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, b);
    }
    valid = valid && !__any_sync(0xffffffffu, bad) && !aborted;
    auto row_of = [&](int c) -> long long {
      return (static_cast<long long>(b) * a.nq + c / a.g) * a.Hq + h * a.g + c % a.g;
    };
    float o[8][2][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int ct = 0; ct < 2; ++ct)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][ct][e] = 0.0f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
    if (valid && ng > 0) {
      const int c_lo = 16 * tile + gi, c_hi = c_lo + 8;
      uint32_t qa[8][4];   // A operand: columns c_lo (rows gi), c_hi (rows gi + 8); channels 16 kk + 2 ti (+1, +8, +9)
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
#pragma unroll
        for (int e = 0; e < 4; ++e) qa[kk][e] = 0u;
      if (colw) {
        const uint32_t* qlo = c_lo < cols ? reinterpret_cast<const uint32_t*>(a.q + row_of(c_lo) * kD) : nullptr;
        const uint32_t* qhi = c_hi < cols ? reinterpret_cast<const uint32_t*>(a.q + row_of(c_hi) * kD) : nullptr;
        auto f16w = [&](uint32_t w) -> uint32_t {   // two query values as f16x2 (bf16 widened, then rounded: exact)
          if (a.dtype == S4KV_F16) return w;
          return pack_f16x2(widen16(static_cast<uint16_t>(w & 0xffff), S4KV_BF16),
                            widen16(static_cast<uint16_t>(w >> 16), S4KV_BF16));
        };
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int wc = 8 * kk + ti;   // word of channels 16 kk + 2 ti, + 1
          if (qlo) {
            qa[kk][0] = f16w(qlo[wc]);
            qa[kk][2] = f16w(qlo[wc + 4]);
          }
          if (qhi) {
            qa[kk][1] = f16w(qhi[wc]);
            qa[kk][3] = f16w(qhi[wc + 4]);
          }
        }
      }
      const int lim_lo = c_lo < cols ? T - a.nq + c_lo / a.g + 1 : T;
      const int lim_hi = c_hi < cols ? T - a.nq + c_hi / a.g + 1 : T;
      int free_end = min(lim_lo, lim_hi);   // groups ending at or before it need no mask
#pragma unroll
      for (int x = 1; x < 32; x <<= 1) free_end = min(free_end, __shfl_xor_sync(0xffffffffu, free_end, x));
      const uint32_t khi_s = smem_u32(blk + M::kKhi), klo_s = smem_u32(blk + M::kKlo), vt_s = smem_u32(blk + M::kVt);
      auto issue = [&](int s, int i) {   // leader: the records of group i into stage s
        const int g = group_of(i);
        const int np = 32 * g + kP < T ? 2 : 1;
        const int p0 = sg.bt[2 * g], p1 = np == 2 ? sg.bt[2 * g + 1] : p0;
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          char* dst = blk + s * M::kStage;
          mbar_expect_tx(&full[s], np * F::kBytes);
          bulk_load_hint(dst, rec_at<BITS>(sg, p0), F::kBytes, &full[s], once);
          if (np == 2) bulk_load_hint(dst + kRecStrideB<BITS>, rec_at<BITS>(sg, p1), F::kBytes, &full[s], once);
        }
        pend |= 1u << s;
      };
      if (leader) {
        for (int i = 0; i < ng && i < 2; ++i) issue(i, i);
      }
      for (int i = 0; i < ng; ++i) {
        const int s = i & 1;
        if (leader) {
          const bool got = __all_sync(0xffffffffu, mbar_wait(&full[s], (fph >> s) & 1u, a.wait_ns));
          if (got) {
            fph ^= 1u << s;
            pend &= ~(1u << s);
          }
          if (lane == 0) team_ok[team] = got ? 1 : 0;
        }
        team_sync();
        if (!team_ok[team]) {   // the same outcome for every warp of the team
          aborted = true;
          break;
        }
        if (!leader) {   // the phase has completed: this wait orders the records' bytes for this warp
          mbar_wait(&full[s], (fph >> s) & 1u, kDrainNs);
          fph ^= 1u << s;
        }
        const int g = group_of(i), t0 = 32 * g;
        const char* stage = blk + s * M::kStage;
        if (t0 + kG <= min(Tk, Tv)) {
          restore_keys<BITS, false>(stage, blk + M::kKhi, blk + M::kKlo, t0, T, Tk, kring, a.dtype, thr, nthr);
          restore_values<BITS, false>(stage, blk + M::kVt, t0, T, Tv, vring, a.R, a.dtype, thr, nthr);
        } else {
          restore_keys<BITS, true>(stage, blk + M::kKhi, blk + M::kKlo, t0, T, Tk, kring, a.dtype, thr, nthr);
          restore_values<BITS, true>(stage, blk + M::kVt, t0, T, Tv, vring, a.R, a.dtype, thr, nthr);
        }
        fence_proxy_async();   // the stage's generic reads come before its next bulk copy
        team_sync();
        if (leader && i + 2 < ng) issue(s, i + 2);
        if (colw) {
          const float scale = a.sm_scale_log2;
          if (t0 + kG > free_end) mq_group_mma<true>(khi_s, klo_s, vt_s, o, m, l, qa, scale, t0, lim_lo, lim_hi);
          else mq_group_mma<false>(khi_s, klo_s, vt_s, o, m, l, qa, scale, t0, lim_lo, lim_hi);
        }
        team_sync();   // the restored group is free again
      }
      if (aborted) {
        if (leader) {
          if (lane == 0) report(a.status, S4KV_ERR_DEVICE_TIMEOUT, S4KV_DEV_TIMEOUT, b);
          for (int s = 0; s < 2; ++s) {
            if ((pend >> s) & 1u) {
              mbar_wait(&full[s], (fph >> s) & 1u, kDrainNs);
              fph ^= 1u << s;
              pend &= ~(1u << s);
            }
          }
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int ct = 0; ct < 2; ++ct)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][ct][e] = 0.0f;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.0f;
      }
    }
    // every warp passes these two barriers once per segment: the team is done with
    // the stages and the restored group before warps write scratch in their regions
    team_sync();
#pragma unroll
    for (int rw = 0; rw < 2; ++rw) {
      l[rw] += __shfl_xor_sync(0xffffffffu, l[rw], 1);
      l[rw] += __shfl_xor_sync(0xffffffffu, l[rw], 2);
    }
    if (leader && seg_start >= r0 && lane == 0) {
      int ncon = 0;
      if (!own && slot_ok) ncon = owner_of(seg_end - 1, C, n_act) - gteam + 1;
      const long long first = 2LL * gteam + (seg_start <= r0 ? 0 : 1);
      meta_of(a)[static_cast<long long>(b) * a.H + h] =
          static_cast<long long>(static_cast<unsigned>(first)) | (static_cast<long long>(ncon) << 32);
    }
    if (colw) {
#pragma unroll
      for (int ct = 0; ct < 2; ++ct) {
        MmaState ms;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) ms.o[mt][e] = o[mt][ct][e];
#pragma unroll
        for (int k = 0; k < 4; ++k) ms.bias[k] = 0.0f;
        ms.m0 = __shfl_sync(0xffffffffu, m[ct], 8 * ti);
        ms.m1 = __shfl_sync(0xffffffffu, m[ct], 8 * ti + 4);
        const float lt0 = __shfl_sync(0xffffffffu, l[ct], 8 * ti), lt1 = __shfl_sync(0xffffffffu, l[ct], 8 * ti + 4);
        ms.l0 = lane < 4 ? lt0 : 0.0f;
        ms.l1 = lane < 4 ? lt1 : 0.0f;
        GenState gs;
        mma_to_gen(ms, gs, scratch);
        if (own || !slot_ok) {
#pragma unroll
          for (int jj = 0; jj < kNH; ++jj) {
            const int c = 16 * tile + 8 * ct + jj;
            if (c < cols) {
              const float inv = gs.l[jj] > 0.0f ? 1.0f / gs.l[jj] : 0.0f;
              store_out(a, row_of(c), lane,
                        make_float4(gs.o[jj][0] * inv, gs.o[jj][1] * inv, gs.o[jj][2] * inv, gs.o[jj][3] * inv));
            }
          }
        } else {
          const int k = seg_start <= r0 ? 0 : 1;
          float* P = a.ws + (2LL * gw + k) * partial_floats(a.pcols);
#pragma unroll
          for (int jj = 0; jj < kNH; ++jj) {
            const int cc = 8 * ct + jj;
            *reinterpret_cast<float4*>(P + cc * kD + 4 * lane) =
                make_float4(gs.o[jj][0], gs.o[jj][1], gs.o[jj][2], gs.o[jj][3]);
            if (lane == 0) {
              P[a.pcols * kD + 2 * cc] = gs.m[jj];
              P[a.pcols * kD + 2 * cc + 1] = gs.l[jj];
            }
          }
        }
      }
    }
    fence_proxy_async();   // the scratch writes come before later bulk copies into the region
    team_sync();
    seg_start = seg_end;
    if (++h == a.H) {
      h = 0;
      if (++b >= a.B) break;
      sc = seg_cost(a.seq_lens[b], a.R, a.tail_cost);
    }
  }
  if (pend) {   // never expected: every issued copy is waited for
    for (int s = 0; s < 2; ++s)
      if ((pend >> s) & 1u) mbar_wait(&full[s], (fph >> s) & 1u, kDrainNs);
  }
}

// Multi-query attention over KIVI pages on tcgen05, warp-specialized. The CTA is
// one team and works through its slice of the cost line segment by segment:
//  * warps 4 .. 10 restore each key group into one of two slots of core-matrix
//    tiles (K^ high and low, V^) and stage page records two groups ahead;
//  * warp 11 issues the MMAs: S[slot] = Q K^T (M = 128 query columns, N = 32
//    tokens, K = 128) into one of two tensor-memory buffers once a slot is
//    restored, and O += P V (N = 128 channels, K = 32 tokens) once P is written;
//  * warps 0 .. 3 read S one query column per thread (TMEM lane), run the lazy
//    online softmax, rescale their O rows in tensor memory when the maximum moves,
//    and write P.
// Hand-offs are mbarriers (tcgen05.commit for the MMAs) waited on with a bound; a
// wait that runs out raises a shared flag and every role leaves its loop. The only
// CTA-wide barriers sit between the roles' loops, reached by every thread once per
// segment; the mbarriers are re-initialised between segments, when nothing is in
// flight. Tensor memory is allocated after the CTA-uniform exit and freed on the
// only way out.
template <int BITS>
__global__ void __launch_bounds__(32 * S4KV_DECODE_WARPS, 1) mqt_kernel(DecodeArgs a) {
  constexpr int kWarps = S4KV_DECODE_WARPS;
  constexpr int kThreads = 32 * kWarps;
  static_assert(kWarps == 12, "4 softmax warps, 7 restoring warps and an MMA warp");
  constexpr int kProd0 = 4, kProdWarps = 7, kMmaWarp = 11;
  using F = Rec<BITS>;
  using SmemT = Smem<kWarps>;
  constexpr int kStage = kStageBytesB<BITS>;
  constexpr int kRecStages = 4, kSlots = 3;               // records staged ahead; restored groups in flight
  constexpr int kQ = (kRecStages * kStage + 1023) / 1024 * 1024;   // Q: 128 columns x 128 channels
  constexpr int kTile = kG * kD * 2;                       // one 32 x 128 f16 tile
  constexpr int kSlot0 = kQ + 128 * kD * 2;                // slot s at kSlot0 + 3 s kTile: K^ hi, K^ lo, V^
  constexpr int kPo = kSlot0 + 3 * kSlots * kTile;         // P: 128 columns x 32 tokens
  static_assert(kPo + 128 * kG * 2 <= kWarps * kRegion, "tiles fit the CTA's regions");
  constexpr uint32_t kTmemCols = 256;                      // O in columns 0 .. 127, S[s] at 128 + 32 s
  static_assert(128 + 32 * kSlots <= static_cast<int>(kTmemCols), "S buffers fit the allocation");
  enum { kRecFull = 0, kSlotReady = kRecStages, kSFull = kSlotReady + kSlots, kSlotFree = kSFull + kSlots,
         kPReady = kSlotFree + kSlots, kPvDone = kPReady + 1, kNumBars = kPvDone + 1 };
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmemT& sm = *reinterpret_cast<SmemT*>(smem_raw);
  long long* pre = reinterpret_cast<long long*>(smem_raw + prefix_offset<0>());   // [B + 1]
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t bars[kNumBars];
  __shared__ int abort_flag;
  char* base = reinterpret_cast<char*>(sm.region[0]);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto init_bars = [&]() {   // thread 0
    for (int k = 0; k < kRecStages; ++k) mbar_init(&bars[kRecFull + k], 1);
    for (int k = 0; k < kSlots; ++k) {
      mbar_init(&bars[kSlotReady + k], kProdWarps);
      mbar_init(&bars[kSFull + k], 1);
      mbar_init(&bars[kSlotFree + k], 1);
    }
    mbar_init(&bars[kPReady], 4);
    mbar_init(&bars[kPvDone], 1);
  };
  {
    long long carry = 0;
    __shared__ long long wt[kWarps];
    for (int base_b = 0; base_b < a.B; base_b += kThreads) {
      const int b = base_b + tid;
      const long long cnt = b < a.B ? a.H * seg_cost(a.seq_lens[b], a.R, a.tail_cost).cost : 0;
      long long x = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) wt[warp] = x;
      __syncthreads();
      long long before = carry, total = 0;
      for (int q = 0; q < kWarps; ++q) {
        if (q < warp) before += wt[q];
        total += wt[q];
      }
      if (b < a.B) pre[b] = before + x - cnt;
      __syncthreads();
      carry += total;
    }
    if (tid == 0) pre[a.B] = carry;
    __syncthreads();
  }
  const long long C = pre[a.B];
  int n_act = static_cast<int>(gridDim.x);   // one team per CTA
  if (a.max_warps > 0 && a.max_warps < n_act) n_act = a.max_warps;
  {
    const long long cap = (C + kMinUnits - 1) / kMinUnits;
    if (cap < n_act) n_act = static_cast<int>(cap);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int gteam = blockIdx.x;
  if (gteam >= n_act) return;   // CTA-uniform, before tensor memory is allocated

  if (tid == 0) {
    init_bars();
    abort_flag = 0;
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "n"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t t_row = static_cast<uint32_t>(32 * (warp & 3)) << 16;   // softmax warp's TMEM lanes
  volatile int* flag = &abort_flag;

  const long long r0 = gteam * C / n_act, r1 = (gteam + 1) * C / n_act;
  const uint64_t once = policy_evict_first();
  const int cols = a.nq * a.g;
  const float scale = a.sm_scale_log2;
  const uint32_t q_s = smem_u32(base + kQ), p_s = smem_u32(base + kPo);
  uint32_t ph = 0;     // this thread's phase bit of each mbarrier
  uint32_t pend = 0;   // warp kProd0: record copies in flight
  bool aborted = false;
  // warp-uniform bounded wait; false (and the flag raised) when it runs out or the
  // flag is already up
  // tracing builds: per warp [0] span, [1] first wait, [2] second wait, [3] work, [4] groups
  S4KV_TRACE(unsigned long long tq[5] = {global_ns(), 0, 0, 0, 0}; unsigned long long tmark = 0;)
  auto wait_w = [&](int k) -> bool {
    if (__shfl_sync(0xffffffffu, *flag, 0)) return false;
    const bool ok = __all_sync(0xffffffffu, mbar_wait_sleep(&bars[k], (ph >> k) & 1u, a.wait_ns));
    if (ok) ph ^= 1u << k;
    else if (lane == 0) *flag = 1;
    return ok;
  };

  int b;
  {
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  SegCost sc = seg_cost(a.seq_lens[b], a.R, a.tail_cost);
  int h = static_cast<int>((r0 - pre[b]) / sc.cost);
  long long seg_start = pre[b] + h * sc.cost;

  while (seg_start < r1) {
    const long long seg_end = seg_start + sc.cost;
    const int T = max(a.seq_lens[b], 0);
    const long long lo = max(r0, seg_start) - seg_start, hi = min(r1, seg_end) - seg_start;
    const bool own = lo == 0 && hi == sc.cost;
    const int nm = sc.main_groups;
    const int u0 = static_cast<int>(lo < nm ? lo : nm), u1 = static_cast<int>(hi < nm ? hi : nm);
    int c0 = 0, c1 = 0;
    if (sc.tail_chunks > 0 && hi > nm) {
      c0 = static_cast<int>(lo > nm ? (lo - nm + a.tail_cost - 1) / a.tail_cost : 0);
      const long long cc = (hi - nm + a.tail_cost - 1) / a.tail_cost;
      c1 = static_cast<int>(cc < sc.tail_chunks ? cc : sc.tail_chunks);
    }
    const int nmain = u1 - u0, ng = nmain + (c1 - c0);
    auto group_of = [&](int i) { return i < nmain ? u0 + i : nm + c0 + (i - nmain); };
    const int slot = a.slot_ids ? a.slot_ids[b] : b;
    const bool slot_ok = slot >= 0 && slot < a.max_slots;
    const bool table_ok = static_cast<long long>(a.bt_stride) * kP >= T;
    const int lens_v = slot_ok ? a.lens[slot * a.H + h] : 0;
    Seg sg;
    sg.pages = a.pages;
    sg.bt = a.block_table + static_cast<long long>(b) * a.bt_stride;
    sg.H = a.H;
    sg.h = h;
    sg.T = T;
    const int npT = (T + kP - 1) / kP;
    const int Tk = T & ~(kG - 1), Tv = max(0, T - a.R);
    const uint16_t* kring = reinterpret_cast<const uint16_t*>(a.kring) + (slot_ok ? slot : 0) * a.kring_slot + h * a.kring_head;
    const uint16_t* vring = reinterpret_cast<const uint16_t*>(a.vring) + (slot_ok ? slot : 0) * a.vring_slot + h * a.vring_head;
    bool valid = slot_ok && T > 0;
    bool bad = false;
    if (warp == 0 && valid && table_ok && ng > 0) {
      const int p_lo = 2 * group_of(0), p_hi = min(2 * group_of(ng - 1) + 2, npT);
      for (int pb = p_lo; pb < p_hi; pb += 32 * 8) {
        int pp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int lp = pb + 32 * k + lane;
          pp[k] = lp < p_hi ? sg.bt[lp] : 0;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (pb + 32 * k + lane < p_hi && (pp[k] < 0 || pp[k] >= a.num_pages)) {
            bad = true;
            report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp[k]);
          }
        }
      }
    }
    if (!slot_ok) {
      if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
    } else if (lens_v != T || T > a.max_seq_len || T < a.nq) {
      valid = false;
      if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, b);
    } else if (!table_ok) {
      valid = false;
      if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, b);
    }
    valid = !__syncthreads_or(bad) && valid && !aborted;   // the same for every thread
    auto row_of = [&](int c) -> long long {
      return (static_cast<long long>(b) * a.nq + c / a.g) * a.Hq + h * a.g + c % a.g;
    };
    const int r = tid;   // softmax warps: query column of this thread
    const int lim = r < cols ? T - a.nq + r / a.g + 1 : T;
    const int free_end = T - a.nq + 1;   // groups ending by then need no causal mask
    float m_r = -INFINITY, l_r = 0.0f;
    ph = 0;   // the mbarriers start this segment freshly initialised
    if (valid && ng > 0) {
      for (int it = tid; it < 128 * 16; it += kThreads) {   // Q: zero past cols
        const int row = it & 127, c0q = 8 * (it >> 7);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < cols) {
          v = *reinterpret_cast<const uint4*>(a.q + row_of(row) * kD + c0q);
          if (a.dtype == S4KV_BF16) {
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
              w[k] = pack_f16x2(widen16(static_cast<uint16_t>(w[k] & 0xffff), S4KV_BF16),
                                widen16(static_cast<uint16_t>(w[k] >> 16), S4KV_BF16));
            v = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        *reinterpret_cast<uint4*>(base + kQ + core_off(row, c0q, kCoreSbo128)) = v;
      }
      fence_proxy_async();
      __syncthreads();
      auto issue = [&](int s, int i) {   // warp kProd0: the records of group i into record stage s
        const int g = group_of(i);
        const int np = 32 * g + kP < T ? 2 : 1;
        const int p0 = sg.bt[2 * g], p1 = np == 2 ? sg.bt[2 * g + 1] : p0;
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          char* dst = base + s * kStage;
          mbar_expect_tx(&bars[kRecFull + s], np * F::kBytes);
          bulk_load_hint(dst, rec_at<BITS>(sg, p0), F::kBytes, &bars[kRecFull + s], once);
          if (np == 2) bulk_load_hint(dst + kRecStrideB<BITS>, rec_at<BITS>(sg, p1), F::kBytes, &bars[kRecFull + s], once);
        }
        pend |= 1u << s;
      };
      if (warp >= kProd0 && warp < kProd0 + kProdWarps) {
        // ---- restoring warps ----
        const int pt = tid - 32 * kProd0, npt = 32 * kProdWarps;
        if (warp == kProd0) {
          for (int i = 0; i < ng && i < kRecStages; ++i) issue(i, i);
        }
        for (int i = 0; i < ng; ++i) {
          const int s = i % kSlots, rs = i % kRecStages;
          S4KV_TRACE(tmark = global_ns();)
          if (i >= kSlots && !wait_w(kSlotFree + s)) break;   // P V of group i - kSlots done with slot s
          S4KV_TRACE({ const unsigned long long x = global_ns(); tq[1] += x - tmark; tmark = x; })
          if (!wait_w(kRecFull + rs)) break;
          S4KV_TRACE({ const unsigned long long x = global_ns(); tq[2] += x - tmark; tmark = x; })
          if (warp == kProd0) pend &= ~(1u << rs);
          const int g = group_of(i), t0 = 32 * g;
          const char* stage = base + rs * kStage;
          char* tiles = base + kSlot0 + 3 * s * kTile;
          if (t0 + kG <= min(Tk, Tv)) {
            restore_keys<BITS, false, true>(stage, tiles, tiles + kTile, t0, T, Tk, kring, a.dtype, pt, npt);
            restore_values<BITS, false, true>(stage, tiles + 2 * kTile, t0, T, Tv, vring, a.R, a.dtype, pt, npt);
          } else {
            restore_keys<BITS, true, true>(stage, tiles, tiles + kTile, t0, T, Tk, kring, a.dtype, pt, npt);
            restore_values<BITS, true, true>(stage, tiles + 2 * kTile, t0, T, Tv, vring, a.R, a.dtype, pt, npt);
          }
          fence_proxy_async();   // tile writes before the MMAs; stage reads before its next copy
          __syncwarp();
          if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bars[kSlotReady + s])) : "memory");
          S4KV_TRACE(tq[3] += global_ns() - tmark; tq[4] += 1;)
          if (warp == kProd0 && i + kRecStages < ng) {
            if (!wait_w(kSlotReady + s)) break;   // every restoring warp is done with record stage rs
            issue(rs, i + kRecStages);
          }
        }
      } else if (warp == kMmaWarp) {
        // ---- MMA warp ----
        auto pv = [&](int i) {   // O += P V of group i (slot i % kSlots)
          tc_fence_after();
          if (lane == 0) {
            const uint32_t v_s = smem_u32(base + kSlot0 + 3 * (i % kSlots) * kTile + 2 * kTile);
#pragma unroll
            for (int j = 0; j < 2; ++j)
              umma_f16(tmem, umma_desc(p_s + 256 * j, kCoreSbo32), umma_desc(v_s + 256 * j, kCoreSbo32),
                       umma_idesc(128, kD), i > 0 || j > 0);
            umma_commit(&bars[kSlotFree + i % kSlots]);
            umma_commit(&bars[kPvDone]);
          }
          __syncwarp();
        };
        bool ok = true;
        for (int i = 0; i < ng && ok; ++i) {
          const int s = i % kSlots;
          S4KV_TRACE(tmark = global_ns();)
          if (!wait_w(kSlotReady + s)) { ok = false; break; }
          S4KV_TRACE({ const unsigned long long x = global_ns(); tq[1] += x - tmark; tq[4] += 1; })
          tc_fence_after();
          if (lane == 0) {
            const uint32_t kh_s = smem_u32(base + kSlot0 + 3 * s * kTile), kl_s = kh_s + kTile;
            const uint32_t d = tmem + 128 + 32 * s;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              umma_f16(d, umma_desc(q_s + 256 * j, kCoreSbo128), umma_desc(kh_s + 256 * j, kCoreSbo128),
                       umma_idesc(128, kG), j > 0);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              umma_f16(d, umma_desc(q_s + 256 * j, kCoreSbo128), umma_desc(kl_s + 256 * j, kCoreSbo128),
                       umma_idesc(128, kG), true);
            umma_commit(&bars[kSFull + s]);
          }
          __syncwarp();
          if (i >= 1) {
            S4KV_TRACE(tmark = global_ns();)
            if (!wait_w(kPReady)) { ok = false; break; }
            S4KV_TRACE(tq[2] += global_ns() - tmark;)
            pv(i - 1);
          }
        }
        if (ok && wait_w(kPReady)) pv(ng - 1);
      } else if (warp < 4) {
        // ---- softmax warps ----
        bool ok = true;
        for (int i = 0; i < ng; ++i) {
          const int s = i % kSlots;
          S4KV_TRACE(tmark = global_ns();)
          if (!wait_w(kSFull + s)) { ok = false; break; }
          S4KV_TRACE({ const unsigned long long x = global_ns(); tq[1] += x - tmark; tmark = x; tq[4] += 1; })
          tc_fence_after();
          uint32_t sr[32];
          tmem_ld32(tmem + t_row + 128 + 32 * s, sr);
          tmem_wait_ld();
          const int t0 = 32 * group_of(i);
          const bool mask = t0 + kG > free_end;
          float z[32];
          float mx = -INFINITY;
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            z[x] = __uint_as_float(sr[x]) * scale;
            if (mask && t0 + x >= lim) z[x] = -INFINITY;
            mx = fmaxf(mx, z[x]);
          }
          if (i >= 1) {   // P V of group i - 1 done: P is free and O holds groups < i
            S4KV_TRACE({ const unsigned long long x = global_ns(); tq[3] += x - tmark; tmark = x; })
            if (!wait_w(kPvDone)) { ok = false; break; }
            S4KV_TRACE({ const unsigned long long x = global_ns(); tq[2] += x - tmark; tmark = x; })
            tc_fence_after();
          }
          const bool need = mx > m_r + kLazy;
          if (__any_sync(0xffffffffu, need)) {
            const float mn = need ? mx : m_r;
            const float al = (!need || mn == -INFINITY) ? 1.0f : ex2(m_r - mn);
            m_r = mn;
            l_r *= al;
            if (i >= 1) {   // O already holds earlier groups: rescale this column's row
#pragma unroll 1
              for (int ch = 0; ch < 4; ++ch) {
                uint32_t orow[32];
                tmem_ld32(tmem + t_row + 32 * ch, orow);
                tmem_wait_ld();
#pragma unroll
                for (int x = 0; x < 32; ++x) orow[x] = __float_as_uint(__uint_as_float(orow[x]) * al);
                tmem_st32(tmem + t_row + 32 * ch, orow);
              }
              tmem_wait_st();
            }
          }
          uint32_t pk[16];
          float sum = 0.0f;
#pragma unroll
          for (int x = 0; x < 32; x += 2) {
            const float p0 = z[x] == -INFINITY ? 0.0f : ex2(z[x] - m_r);
            const float p1 = z[x + 1] == -INFINITY ? 0.0f : ex2(z[x + 1] - m_r);
            sum += p0 + p1;
            pk[x >> 1] = pack_f16x2(p0, p1);
          }
          l_r += sum;
#pragma unroll
          for (int kg = 0; kg < 4; ++kg)
            *reinterpret_cast<uint4*>(base + kPo + core_off(r, 8 * kg, kCoreSbo32)) =
                make_uint4(pk[4 * kg], pk[4 * kg + 1], pk[4 * kg + 2], pk[4 * kg + 3]);
          fence_proxy_async();   // P's generic writes before the MMA reads them
          tc_fence_before();
          __syncwarp();
          if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bars[kPReady])) : "memory");
          S4KV_TRACE(tq[3] += global_ns() - tmark;)
        }
        if (ok && wait_w(kPvDone)) tc_fence_after();   // the last P V: O is final
      }
    }
    __syncthreads();   // every role has left its loop
    aborted = *flag != 0;
    if (aborted && warp == kProd0) {   // drain record copies still in flight
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE_TIMEOUT, S4KV_DEV_TIMEOUT, b);
      for (int s = 0; s < kRecStages; ++s)
        if ((pend >> s) & 1u) mbar_wait(&bars[kRecFull + s], (ph >> (kRecFull + s)) & 1u, kDrainNs);
      pend = 0;
    }
    if (tid == 0 && seg_start >= r0) {
      int ncon = 0;
      if (!own && slot_ok) ncon = owner_of(seg_end - 1, C, n_act) - gteam + 1;
      const long long first = 2LL * gteam + (seg_start <= r0 ? 0 : 1);
      meta_of(a)[static_cast<long long>(b) * a.H + h] =
          static_cast<long long>(static_cast<unsigned>(first)) | (static_cast<long long>(ncon) << 32);
    }
    if (warp < 4) {
      const bool have = valid && ng > 0 && !aborted;   // the same for every thread
      if (!have) {
        m_r = -INFINITY;
        l_r = 0.0f;
      }
      const float inv = l_r > 0.0f ? 1.0f / l_r : 0.0f;
      const int k = seg_start <= r0 ? 0 : 1;
      float* part = a.ws + (2LL * (static_cast<long long>(gteam) * kWarps + r / 16) + k) * partial_floats(a.pcols);
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t orow[32];
        if (have) {
          tmem_ld32(tmem + t_row + 32 * ch, orow);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) orow[x] = 0u;
        }
        if (r < cols) {
          if (own || !slot_ok) {
#pragma unroll
            for (int x = 0; x < 32; x += 4)
              store_out(a, row_of(r), (32 * ch + x) / 4,
                        make_float4(__uint_as_float(orow[x]) * inv, __uint_as_float(orow[x + 1]) * inv,
                                    __uint_as_float(orow[x + 2]) * inv, __uint_as_float(orow[x + 3]) * inv));
          } else {
#pragma unroll
            for (int x = 0; x < 32; x += 4)
              *reinterpret_cast<float4*>(part + (r % 16) * kD + 32 * ch + x) =
                  make_float4(__uint_as_float(orow[x]), __uint_as_float(orow[x + 1]), __uint_as_float(orow[x + 2]),
                              __uint_as_float(orow[x + 3]));
          }
        }
      }
      if (r < cols && !(own || !slot_ok)) {
        part[a.pcols * kD + 2 * (r % 16)] = m_r;
        part[a.pcols * kD + 2 * (r % 16) + 1] = l_r;
      }
    }
    if (tid == 0 && !aborted && valid && ng > 0) {   // nothing is in flight: fresh barriers for the next segment
      for (int k = 0; k < kNumBars; ++k) asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(&bars[k])) : "memory");
      init_bars();
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tc_fence_before();
    __syncthreads();   // O, Q, P and the slots are free for the next segment
    tc_fence_after();
    seg_start = seg_end;
    if (++h == a.H) {
      h = 0;
      if (++b >= a.B) break;
      sc = seg_cost(a.seq_lens[b], a.R, a.tail_cost);
    }
  }
  S4KV_TRACE({
    if (lane == 0) {
      unsigned long long* out = reinterpret_cast<unsigned long long*>(meta_of(a) + meta_words(a.B, a.H)) +
                                (static_cast<long long>(blockIdx.x) * kWarps + warp) * kTraceWords;
      out[0] = global_ns() - tq[0];
      for (int k = 1; k < 5; ++k) out[k] = tq[k];
    }
  })
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols));
}

// Merge for mq_kernel: one warp per (segment, column). Contributor i of a
// segment is team slot first + ... as in merge_kernel; the warp of column c in
// team t is warp (t / tpc) * kWarps + (t % tpc) * tw + c / 8 of the grid.
__global__ void __launch_bounds__(32 * kMergeWarps) mq_merge_kernel(DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int kWarps = S4KV_DECODE_WARPS;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long* desc = meta_of(a);
  const int cols = a.nq * a.g, tpc = kWarps / a.tw;
  const long long items = static_cast<long long>(a.B) * a.H * cols;
  const long long pf = partial_floats(a.pcols);
  for (long long it = static_cast<long long>(blockIdx.x) * kMergeWarps + warp; it < items;
       it += static_cast<long long>(gridDim.x) * kMergeWarps) {
    const int c = static_cast<int>(it % cols);
    const long long bh = it / cols;
    const long long d = __ldcg(desc + bh);
    const int nc = static_cast<int>(d >> 32);
    if (nc <= 0) continue;
    const long long first = static_cast<long long>(static_cast<unsigned>(d & 0xffffffffLL));
    const int tile = c / a.pcols, col = c % a.pcols;   // a warp holds pcols columns
    auto part = [&](int i) -> const float* {
      const long long ts = i == 0 ? first : (first & ~1LL) + 2LL * i;
      const long long gt = ts >> 1;
      const long long gwp = (gt / tpc) * kWarps + (gt % tpc) * a.tw + tile;
      return a.ws + (2LL * gwp + (ts & 1)) * pf;
    };
    float M = -INFINITY, L = 0.0f;
    float4 O = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int i0 = 0; i0 < nc; i0 += kMC) {
      const int nch = min(kMC, nc - i0);
      const float* W = part(i0 + (lane < nch ? lane : 0)) + a.pcols * kD + 2 * col;
      const float mi = lane < nch ? __ldcg(W) : -INFINITY;
      const float li = lane < nch ? __ldcg(W + 1) : 0.0f;
      float4 r[kMC];
#pragma unroll
      for (int u = 0; u < kMC; ++u)
        r[u] = u < nch ? __ldcg(reinterpret_cast<const float4*>(part(i0 + u) + col * kD + 4 * lane))
                       : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      const float mn = fmaxf(M, warp_max(mi));
      const bool live = mn != -INFINITY;
      const float ao = live ? ex2(M - mn) : 1.0f;
      const float wi = live ? ex2(mi - mn) : 0.0f;
      L = fmaf(L, ao, warp_sum(wi * li));
      O = make_float4(O.x * ao, O.y * ao, O.z * ao, O.w * ao);
#pragma unroll
      for (int u = 0; u < kMC; ++u) {
        const float w = __shfl_sync(0xffffffffu, wi, u);
        O = make_float4(fmaf(w, r[u].x, O.x), fmaf(w, r[u].y, O.y), fmaf(w, r[u].z, O.z), fmaf(w, r[u].w, O.w));
      }
      M = mn;
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    const int b = static_cast<int>(bh / a.H), h = static_cast<int>(bh % a.H);
    store_out(a, (static_cast<long long>(b) * a.nq + c / a.g) * a.Hq + h * a.g + c % a.g, lane,
              make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
  }
}

}  // namespace

size_t decode_meta_bytes(int B, int H) { return static_cast<size_t>(meta_words(B, H)) * sizeof(long long); }

int decode_threads(int impl) { return 32 * (impl == 1 ? warps_of<1>() : warps_of<0>()); }
int decode_warps_per_cta(int impl) { return impl == 1 ? warps_of<1>() : warps_of<0>(); }
size_t decode_partial_bytes(int g) { return static_cast<size_t>(partial_floats(g)) * sizeof(float); }
size_t decode_trace_bytes_per_warp() { return kTraceWords ? static_cast<size_t>(kTraceWords + 4) * 8 : 0; }

size_t decode_smem_bytes(int impl, int B) {
  const size_t base = impl == 1 ? prefix_offset<1>() : prefix_offset<0>();
  return base + static_cast<size_t>(B + 1) * sizeof(long long);
}

namespace {
// Grants `kernel` the dynamic shared memory it needs (once per size increase).
cudaError_t grant_smem(void (*kernel)(DecodeArgs), size_t need, size_t* granted) {
  if (need <= *granted) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(need));
  if (e != cudaSuccess) {
    cudaGetLastError();   // leave no error behind for the caller's next CUDA call
    return e;
  }
  *granted = need;
  return cudaSuccess;
}

template <int IMPL, int BITS>
cudaError_t prepare(int B, int* per_sm) {
  static size_t attr_bytes = 0;   // largest dynamic shared memory granted so far
  const size_t need = decode_smem_bytes(IMPL, B);
  const cudaError_t e = grant_smem(decode_kernel<IMPL, BITS>, need, &attr_bytes);
  if (e != cudaSuccess) return e;
  if (per_sm)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, decode_kernel<IMPL, BITS>, 32 * warps_of<IMPL>(),
                                                         need);
  return cudaSuccess;
}

// The instantiations: tensor-core path (0), FFMA path (1, 4-bit only), tensor-core
// path with the key split (2), each for 4-bit and 2-bit records; the tensor-core
// path for FP8 records.
cudaError_t prepare_any(int impl, int bits, int B, int* per_sm) {
  if (bits == 8) return prepare<0, 8>(B, per_sm);
  if (bits == 2) return impl == 2 ? prepare<2, 2>(B, per_sm) : prepare<0, 2>(B, per_sm);
  return impl == 1 ? prepare<1, 4>(B, per_sm) : impl == 2 ? prepare<2, 4>(B, per_sm) : prepare<0, 4>(B, per_sm);
}
}  // namespace

namespace {
// Programmatic-dependent launch of a merge kernel right behind the attention kernel.
cudaError_t launch_merge(void (*kernel)(DecodeArgs), const DecodeArgs& a, long long items, int grid, cudaStream_t st) {
  if (items == 0) return cudaSuccess;
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

cudaError_t launch_mq(const DecodeArgs& args, int grid, cudaStream_t st) {
  static size_t attr[7] = {0, 0, 0, 0, 0, 0, 0};
  DecodeArgs a = args;
  const int cols = a.nq * a.g;
  // KIVI pages: narrow calls fold the scales per warp (mq_kernel, 8 columns a warp);
  // wide ones restore each group once per team (mqd_kernel, 16 columns a warp)
  const int choice = a.bits == 8 ? 0 : a.mq_kernel;
  const bool tc = a.bits != 8 && (choice == 3 || (choice == 0 && cols >= S4KV_MQ_TC_MIN_COLS));
  const bool restore = a.bits != 8 && !tc && (choice == 2 || (choice == 0 && cols >= S4KV_MQ_RESTORE_MIN_COLS));
  a.pcols = a.bits == 8 || restore || tc ? 16 : 8;
  a.tw = (cols + a.pcols - 1) / a.pcols;
  if (restore && a.tw < kMqMinTeam) a.tw = kMqMinTeam;   // the team's regions hold a restored group
  if (tc) a.tw = S4KV_DECODE_WARPS;                       // one team per CTA
  void (*kernel)(DecodeArgs) = a.bits == 8 ? mq_fp8_kernel
                               : tc        ? (a.bits == 2 ? mqt_kernel<2> : mqt_kernel<4>)
                               : restore   ? (a.bits == 2 ? mqd_kernel<2> : mqd_kernel<4>)
                                           : (a.bits == 2 ? mq_kernel<2> : mq_kernel<4>);
  const int which = a.bits == 8 ? 0 : (tc ? 5 : restore ? 1 : 3) + (a.bits == 2 ? 1 : 0);
  const size_t smem = decode_smem_bytes(0, a.B);
  cudaError_t e = grant_smem(kernel, smem, &attr[which]);
  if (e != cudaSuccess) return e;
  kernel<<<grid, 32 * S4KV_DECODE_WARPS, smem, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_merge(mq_merge_kernel, a, static_cast<long long>(a.B) * a.H * a.nq * a.g, grid, st);
}

int decode_ctas_per_sm(int impl, int B) {
  int n = 0;
  const cudaError_t e = prepare_any(impl, 4, B, &n);
  return e == cudaSuccess ? n : 0;
}

cudaError_t launch_decode(const DecodeArgs& a, int impl, int grid, cudaStream_t st) {
  const size_t smem = decode_smem_bytes(impl, a.B);
  if (a.bits != 4 && impl == 1) return cudaErrorInvalidValue;   // FFMA path: 4-bit records only
  if (a.bits == 8 && impl != 0) return cudaErrorInvalidValue;
  cudaError_t e = prepare_any(impl, a.bits, a.B, nullptr);
  if (e != cudaSuccess) return e;
  const int threads = 32 * (impl == 1 ? warps_of<1>() : warps_of<0>());
  if (a.bits == 8) {
    decode_kernel<0, 8><<<grid, threads, smem, st>>>(a);
  } else if (a.bits == 2) {
    if (impl == 2) decode_kernel<2, 2><<<grid, threads, smem, st>>>(a);
    else decode_kernel<0, 2><<<grid, threads, smem, st>>>(a);
  } else {
    if (impl == 1) decode_kernel<1, 4><<<grid, threads, smem, st>>>(a);
    else if (impl == 2) decode_kernel<2, 4><<<grid, threads, smem, st>>>(a);
    else decode_kernel<0, 4><<<grid, threads, smem, st>>>(a);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // merge_kernel right behind it, launched programmatically: its blocks may be
  // scheduled while decode_kernel drains and wait for its completion on the device
  return launch_merge(merge_kernel, a, static_cast<long long>(a.B) * a.H * a.g, grid, st);
}

}  // namespace s4kv
