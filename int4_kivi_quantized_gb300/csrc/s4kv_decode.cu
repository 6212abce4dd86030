// Read side of the cache: paged decode attention over the int4 history plus
// the full-precision residual ("4.4 KV Cache 量化", section 2: P = softmax(QK^T
// / sqrt d), output PV; section 3.2: residual and history both take part).
//
// One persistent kernel. Work items are (sequence, kv head, split of S tokens)
// fetched from an atomic counter. Per item, each warp of the CTA takes 32-token
// key groups round-robin: the two page records of a group (3 KiB each, codes and
// fp32 metadata of one kv head) arrive by 1-D bulk TMA into the warp's stage
// ring, guarded by mbarriers with bounded waits. Compute restores nothing to
// HBM ("给 KV cache 减肥", section 3.1: restore happens when the query reads):
//  * tensor-core path: the per-channel key scale is folded into the query
//    (q'_c = q_c s_c, one f16x2 operand per 16-channel slice) and the key min
//    into a per-head bias; nibbles are unpacked to f16 with the magic-number
//    method (integer OR into the mantissa of 1024.0, then subtract) and fed to
//    mma.sync m16n8k16 with tokens as rows and GQA heads as columns. The value
//    side folds the per-token scale into the probabilities (p'_t = p_t s_tk) and
//    the value min into a per-head, per-group bias, with channels as rows.
//  * FFMA path: the same staging with CUDA-core arithmetic, for comparison.
// Tokens past the last group that is quantized for both keys and values (at
// most R + 31) take a per-token path that reads the rings. Each item ends with
// an (m, l, o) partial; the last item of a (sequence, kv head) to finish merges
// them with the log-sum-exp rule and writes the output.

#include "s4kv_common.cuh"

namespace s4kv {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;
constexpr int kStageBytes = 2 * kRec;           // one key group: two page records
constexpr int kNH = kMaxGroup;                  // head slots per kv head (GQA group <= 8)
constexpr long long kDrainNs = 1000000000LL;    // limit for draining copies after a timeout

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

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
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

// Eight nibbles n0..n7 of w to four f16x2 registers holding the exact integer
// codes (n0, n4), (n1, n5), (n2, n6), (n3, n7). OR-ing a nibble into the low
// mantissa bits of 1024.0 (0x6400) gives 1024 + n; a nibble at bits 4..7 gives
// 1024 + 16 n; subtracting (or scaling and subtracting) leaves n exactly.
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

__device__ __forceinline__ float exp2_safe(float x) { return x == -INFINITY ? 0.0f : exp2f(x); }

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

// Float offset of q[h][c..c+3] (c a multiple of 4) in the shared query buffer.
// The 16-byte slots of each head row are XOR-swizzled so that the tensor-core
// path, where lane (gi, ti) reads head gi, channels 32 ti + 4 kk, hits eight
// distinct bank groups per quarter-warp; broadcast readers are unaffected.
__device__ __forceinline__ int q_off(int h, int c) {
  const int s = c >> 2;
  const int phys = (s & ~7) | ((s ^ ((s >> 3) + 4 * (h & 1))) & 7);
  return h * kD + 4 * phys;
}

// ---- per-item context ---------------------------------------------------------------
struct Item {
  const char* pages;   // layer page region
  const int* bt;       // block-table row
  const uint16_t* kring;
  const uint16_t* vring;
  int H, h, T, Tk, Tv, R, dtype, g;
  float scale;         // sm_scale * log2(e)
};

__device__ __forceinline__ const char* rec_of(const Item& it, int logical_page) {
  return it.pages + (static_cast<long long>(it.bt[logical_page]) * it.H + it.h) * kRec;
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
// for absent tokens). Writes p into ptile[token][head].
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
  *reinterpret_cast<float4*>(ptile + lane * kNH) = make_float4(p[0], p[1], p[2], p[3]);
  *reinterpret_cast<float4*>(ptile + lane * kNH + 4) = make_float4(p[4], p[5], p[6], p[7]);
  __syncwarp();
}

// Codes, scale and min of value token tau (page-local) for channels 4l..4l+3,
// from a page record (shared or global memory).
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

__device__ __forceinline__ void gen_pv_token(GenState& s, const float (&v)[4], const float* prow) {
  const float4 p0 = *reinterpret_cast<const float4*>(prow);
  const float4 p1 = *reinterpret_cast<const float4*>(prow + 4);
  const float p[kNH] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
  for (int h = 0; h < kNH; ++h)
#pragma unroll
    for (int q = 0; q < 4; ++q) s.o[h][q] = fmaf(p[h], v[q], s.o[h][q]);
}

// Per-token path for tokens [t0, t0 + n), n <= 32, read straight from pages
// and rings in global memory. Used for the tail past the last fully quantized
// group, and for everything by nothing else.
__device__ void generic_chunk(const Item& it, int t0, int n, GenState& s, float* ptile,
                              const float* q_s) {
  const int lane = threadIdx.x & 31;
  float z[kNH];
#pragma unroll
  for (int h = 0; h < kNH; ++h) z[h] = -INFINITY;
  if (lane < n) {
#pragma unroll
    for (int h = 0; h < kNH; ++h) z[h] = 0.0f;
    const int t = t0 + lane;
    if (t < it.Tk) {
      const char* rec = rec_of(it, t / kP);
      const int tau = t % kP, a = tau & 7, sh = (tau >> 3) * 4;
      const int grp = t / kG;
      const char* m0 = rec_of(it, 2 * grp);
      const char* m1 = rec_of(it, 2 * grp + 1);
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
        const char* mrec = (b >> 1) ? m1 : m0;
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
          const uint4 w4 = *reinterpret_cast<const uint4*>(rec + kKc + kh * 512 + 64 * a + 16 * b);
          const uint32_t wd[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int kq = 0; kq < 4; ++kq) {
            const int kk = 4 * kh + kq, c = 32 * b + 4 * kk;
            const float4 s4 = *reinterpret_cast<const float4*>(mrec + kKm + (2 * kk + (b & 1)) * 16);
            const float4 m4 = *reinterpret_cast<const float4*>(mrec + kKm + (2 * kk + (b & 1)) * 16 + 256);
            const uint32_t w = wd[kq];
            const float k0 = fmaf(code_to_float((w >> sh) & 15u), s4.x, m4.x);
            const float k1 = fmaf(code_to_float((w >> (16 + sh)) & 15u), s4.y, m4.y);
            const float k2 = fmaf(code_to_float((w >> (8 + sh)) & 15u), s4.z, m4.z);
            const float k3 = fmaf(code_to_float((w >> (24 + sh)) & 15u), s4.w, m4.w);
#pragma unroll
            for (int h = 0; h < kNH; ++h) {
              const float4 q4 = *reinterpret_cast<const float4*>(q_s + q_off(h, c));
              z[h] = fmaf(q4.x, k0, fmaf(q4.y, k1, fmaf(q4.z, k2, fmaf(q4.w, k3, z[h]))));
            }
          }
        }
      }
    } else {
      const uint16_t* row = it.kring + static_cast<long long>(t % kG) * kD;
#pragma unroll 1
      for (int c = 0; c < kD; c += 8) {
        const uint4 r4 = *reinterpret_cast<const uint4*>(row + c);
        const uint32_t rw[4] = {r4.x, r4.y, r4.z, r4.w};
        float kv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          kv[2 * i] = widen16(static_cast<uint16_t>(rw[i] & 0xffff), it.dtype);
          kv[2 * i + 1] = widen16(static_cast<uint16_t>(rw[i] >> 16), it.dtype);
        }
#pragma unroll
        for (int h = 0; h < kNH; ++h) {
          const float4 qa = *reinterpret_cast<const float4*>(q_s + q_off(h, c));
          const float4 qb = *reinterpret_cast<const float4*>(q_s + q_off(h, c + 4));
          z[h] = fmaf(qa.x, kv[0], fmaf(qa.y, kv[1], fmaf(qa.z, kv[2], fmaf(qa.w, kv[3], z[h]))));
          z[h] = fmaf(qb.x, kv[4], fmaf(qb.y, kv[5], fmaf(qb.z, kv[6], fmaf(qb.w, kv[7], z[h]))));
        }
      }
    }
#pragma unroll
    for (int h = 0; h < kNH; ++h) z[h] *= it.scale;
  }
  gen_softmax(s, z, ptile);
  for (int tau0 = 0; tau0 < n; tau0 += 4) {
    float v[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = t0 + tau0 + u;
      if (tau0 + u >= n) {
#pragma unroll
        for (int q = 0; q < 4; ++q) v[u][q] = 0.0f;
      } else if (t < it.Tv) {
        value_quad(rec_of(it, t / kP), t % kP, lane, v[u]);
      } else {
        const uint2 r = *reinterpret_cast<const uint2*>(it.vring + static_cast<long long>(t % it.R) * kD + 4 * lane);
        v[u][0] = widen16(static_cast<uint16_t>(r.x & 0xffff), it.dtype);
        v[u][1] = widen16(static_cast<uint16_t>(r.x >> 16), it.dtype);
        v[u][2] = widen16(static_cast<uint16_t>(r.y & 0xffff), it.dtype);
        v[u][3] = widen16(static_cast<uint16_t>(r.y >> 16), it.dtype);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (tau0 + u < n) gen_pv_token(s, v[u], ptile + (tau0 + u) * kNH);
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
    const char* mrec = stage + (lane >> 4) * kRec;
    const int off = kKm + (2 * (lane & 7) + ((lane & 15) >> 3)) * 16;
    const float4 s4 = *reinterpret_cast<const float4*>(mrec + off);
    const float4 m4 = *reinterpret_cast<const float4*>(mrec + off + 256);
#pragma unroll
    for (int h = 0; h < kNH; ++h) {
      const float4 q4 = *reinterpret_cast<const float4*>(q_s + q_off(h, 4 * lane));
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
    const char* rec = stage + (lane >> 4) * kRec;
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
    value_quad(stage + (tau >> 4) * kRec, tau & 15, lane, v);
    gen_pv_token(s, v, ptile + tau * kNH);
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

__device__ void mma_group(const char* stage, MmaState& s, float* ptile, const float* q_s, float scale) {
  const int lane = threadIdx.x & 31, gi = lane >> 2, ti = lane & 3;
  // B operands q'^T for the 8 channel slices, and beta for head gi.
  uint32_t bq0[8], bq1[8];
  float beta = 0.0f;
  {
    const char* mrec = stage + (ti >> 1) * kRec + kKm + (ti & 1) * 16;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const float4 s4 = *reinterpret_cast<const float4*>(mrec + kk * 32);
      const float4 m4 = *reinterpret_cast<const float4*>(mrec + kk * 32 + 256);
      const float4 q4 = *reinterpret_cast<const float4*>(q_s + q_off(gi, 32 * ti + 4 * kk));
      bq0[kk] = pack_f16x2(q4.x * s4.x, q4.y * s4.y);
      bq1[kk] = pack_f16x2(q4.z * s4.z, q4.w * s4.w);
      beta = fmaf(q4.x, m4.x, fmaf(q4.y, m4.y, fmaf(q4.z, m4.z, fmaf(q4.w, m4.w, beta))));
    }
    beta += __shfl_xor_sync(0xffffffffu, beta, 1);
    beta += __shfl_xor_sync(0xffffffffu, beta, 2);
  }
  const float beta0 = __shfl_sync(0xffffffffu, beta, 8 * ti);       // head 2ti
  const float beta1 = __shfl_sync(0xffffffffu, beta, 8 * ti + 4);   // head 2ti+1
  float sc[2][4];
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const char* rec = stage + p * kRec;
    const uint4 w0 = *reinterpret_cast<const uint4*>(rec + kKc + lane * 16);
    const uint4 w1 = *reinterpret_cast<const uint4*>(rec + kKc + 512 + lane * 16);
    const uint32_t wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a[4];
      unpack8(wd[kk], a);
      mma16816(acc, a, bq0[kk], bq1[kk]);
    }
    sc[p][0] = acc[0];
    sc[p][1] = acc[1];
    sc[p][2] = acc[2];
    sc[p][3] = acc[3];
  }
  // online softmax for heads 2ti (even entries) and 2ti+1 (odd entries), in the
  // log2 domain: z = (acc + beta) * scale
  const float bs0 = beta0 * scale, bs1 = beta1 * scale;
  float mx0 = fmaf(fmaxf(fmaxf(sc[0][0], sc[0][2]), fmaxf(sc[1][0], sc[1][2])), scale, bs0);
  float mx1 = fmaf(fmaxf(fmaxf(sc[0][1], sc[0][3]), fmaxf(sc[1][1], sc[1][3])), scale, bs1);
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
  const float off0 = bs0 - s.m0, off1 = bs1 - s.m1;
  float pr[2][4];
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    pr[p][0] = ex2(fmaf(sc[p][0], scale, off0));
    pr[p][1] = ex2(fmaf(sc[p][1], scale, off1));
    pr[p][2] = ex2(fmaf(sc[p][2], scale, off0));
    pr[p][3] = ex2(fmaf(sc[p][3], scale, off1));
    s.l0 += pr[p][0] + pr[p][2];
    s.l1 += pr[p][1] + pr[p][3];
    *reinterpret_cast<float2*>(ptile + (16 * p + gi) * kNH + 2 * ti) = make_float2(pr[p][0], pr[p][1]);
    *reinterpret_cast<float2*>(ptile + (16 * p + gi + 8) * kNH + 2 * ti) = make_float2(pr[p][2], pr[p][3]);
  }
  __syncwarp();
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const char* rec = stage + p * kRec;
    // p for tokens 2ti, 2ti+1, 2ti+8, 2ti+9 of this page, head gi
    const float pe0 = ptile[(16 * p + 2 * ti) * kNH + gi];
    const float pe1 = ptile[(16 * p + 2 * ti + 1) * kNH + gi];
    const float pe2 = ptile[(16 * p + 2 * ti + 8) * kNH + gi];
    const float pe3 = ptile[(16 * p + 2 * ti + 9) * kNH + gi];
    uint32_t b0[4], b1[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 s4 = *reinterpret_cast<const float4*>(rec + kVm + ((2 * k) * 4 + ti) * 16);
      const float4 m4 = *reinterpret_cast<const float4*>(rec + kVm + ((2 * k + 1) * 4 + ti) * 16);
      b0[k] = pack_f16x2(pe0 * s4.x, pe1 * s4.y);
      b1[k] = pack_f16x2(pe2 * s4.z, pe3 * s4.w);
      s.bias[k] = fmaf(pe0, m4.x, fmaf(pe1, m4.y, fmaf(pe2, m4.z, fmaf(pe3, m4.w, s.bias[k]))));
    }
    const uint4 v0 = *reinterpret_cast<const uint4*>(rec + kVc + lane * 16);
    const uint4 v1 = *reinterpret_cast<const uint4*>(rec + kVc + 512 + lane * 16);
    const uint32_t vd[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t a[4];
      unpack8(vd[mt], a);
      mma16816(s.o[mt], a, b0[mt >> 1], b1[mt >> 1]);
    }
  }
  __syncwarp();
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

// ---- the kernel -------------------------------------------------------------------------
struct Smem {
  alignas(128) uint8_t stage[kWarps][kStages][kStageBytes];
  alignas(16) float q_s[kNH * kD];
  alignas(16) float ptile[kWarps][32 * kNH];
  alignas(8) uint64_t bar[kWarps][kStages];
  int item, last, bad, abort_flag;
};

static_assert(sizeof(Smem) % 16 == 0, "shared layout must keep 16-byte alignment");

// Per-warp q' buffers of the FFMA path; the tensor-core path needs none.
template <int IMPL>
__host__ __device__ constexpr size_t extra_bytes() {
  return IMPL == 1 ? sizeof(float) * kWarps * kNH * kD : 0;
}
// Offset of the work-item prefix array (int32 [B + 1]) in dynamic shared memory.
template <int IMPL>
__host__ __device__ constexpr size_t prefix_offset() {
  return (sizeof(Smem) + extra_bytes<IMPL>() + 15) / 16 * 16;
}

__device__ __forceinline__ int nsplit_of(int T, int S) { return T <= 0 ? 1 : (T + S - 1) / S; }

template <int IMPL>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  float* qp_all = reinterpret_cast<float*>(smem_raw + sizeof(Smem));           // FFMA path only
  int* pre = reinterpret_cast<int*>(smem_raw + prefix_offset<IMPL>());         // [B + 1]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(&sm.bar[warp][s], 1);
  }
  if (tid == 0) sm.abort_flag = 0;
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  // prefix of work items: sequence b owns H * nsplit(T_b) items
  {
    int carry = 0;
    for (int base = 0; base < a.B; base += kThreads) {
      const int b = base + tid;
      const int cnt = b < a.B ? a.H * nsplit_of(a.seq_lens[b], a.split) : 0;
      int x = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      __shared__ int wt[kWarps];
      if (lane == 31) wt[warp] = x;
      __syncthreads();
      int before = carry, total = 0;
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
  const int total = pre[a.B];
  const bool ws_ok = total <= a.ws_items;
  if (!ws_ok && blockIdx.x == 0 && tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, total);
  uint32_t issued = 0, consumed = 0;   // per-warp stage counters (warp-uniform)

  while (true) {
    if (tid == 0) sm.item = atomicAdd(a.work, 1);
    if (tid == 0) sm.bad = 0;
    __syncthreads();
    const int item = sm.item;
    if (item >= total) break;
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= item) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int T = max(a.seq_lens[b], 0);
    const int ns = nsplit_of(T, a.split);
    const int r = item - pre[b];
    const int h = r / ns, sp = r % ns;
    const int slot = a.slot_ids ? a.slot_ids[b] : b;
    const int t_lo = sp * a.split, t_hi = min(T, t_lo + a.split);
    const bool slot_ok = slot >= 0 && slot < a.max_slots;
    const bool direct = ns == 1 || !slot_ok || !ws_ok;   // no split-K combine needed
    bool valid = slot_ok && ws_ok;
    if (!slot_ok) {
      if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
    } else if (a.lens[slot * a.H + h] != T) {
      valid = false;
      if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, b);
    } else if (static_cast<long long>(a.bt_stride) * kP < T) {
      valid = false;
      if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, b);
    }
    const int* bt = a.block_table + static_cast<long long>(b) * a.bt_stride;
    if (valid && t_hi > t_lo) {
      // pages this item touches: its own range, plus the group-mates of key metadata
      for (int lp = (t_lo / kG) * 2 + tid; lp < (t_hi + kP - 1) / kP; lp += kThreads) {
        const int pp = bt[lp];
        if (pp < 0 || pp >= a.num_pages) {
          sm.bad = 1;
          report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp);
        }
      }
    }
    for (int i = tid; i < kNH * kD; i += kThreads) {
      const int j = i / kD, c = i % kD;
      sm.q_s[q_off(j, c & ~3) + (c & 3)] =
          (j < a.g) ? widen16(a.q[(static_cast<long long>(b) * a.Hq + h * a.g + j) * kD + c], a.dtype) : 0.0f;
    }
    // order this thread's earlier generic writes to the stage buffers before the
    // bulk copies that will overwrite them
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    valid = valid && !sm.bad && !sm.abort_flag;

    Item it;
    it.pages = a.pages;
    it.bt = bt;
    it.kring = reinterpret_cast<const uint16_t*>(a.kring) + (valid ? slot : 0) * a.kring_slot + h * a.kring_head;
    it.vring = reinterpret_cast<const uint16_t*>(a.vring) + (valid ? slot : 0) * a.vring_slot + h * a.vring_head;
    it.H = a.H;
    it.h = h;
    it.T = T;
    it.Tk = T & ~(kG - 1);
    it.Tv = max(0, T - a.R);
    it.R = a.R;
    it.dtype = a.dtype;
    it.g = a.g;
    it.scale = a.sm_scale_log2;
    const int t_main = min(it.Tk, it.Tv) & ~(kG - 1);

    GenState gs;
    float* ptile = sm.ptile[warp];
    if (valid) {
      const int g_lo = t_lo / kG;
      const int g_hi = max(g_lo, min(t_hi, t_main) / kG);
      // this warp's key groups: g_lo + warp + j * kWarps
      const int my_n = g_hi - g_lo > warp ? (g_hi - g_lo - warp + kWarps - 1) / kWarps : 0;
      auto issue = [&](int j) {
        const int grp = g_lo + warp + j * kWarps;
        const int st = issued % kStages;
        if (lane == 0) {
          uint64_t* bar = &sm.bar[warp][st];
          mbar_expect_tx(bar, kStageBytes);
          bulk_load(sm.stage[warp][st], rec_of(it, 2 * grp), kRec, bar);
          bulk_load(sm.stage[warp][st] + kRec, rec_of(it, 2 * grp + 1), kRec, bar);
        }
        ++issued;
      };
      // next staged group, or -1 when the bounded wait runs out
      auto acquire = [&]() -> int {
        const int st = consumed % kStages;
        if (!mbar_wait(&sm.bar[warp][st], (consumed / kStages) & 1, a.wait_ns)) return -1;
        ++consumed;
        return st;
      };
      int next = 0;
      for (; next < my_n && next < kStages; ++next) issue(next);
      bool ok = true;
      if constexpr (IMPL == 0) {
        MmaState ms;
        mma_init(ms);
        for (int j = 0; j < my_n; ++j) {
          const int st = acquire();
          if (st < 0) { ok = false; break; }
          mma_group(reinterpret_cast<const char*>(sm.stage[warp][st]), ms, ptile, sm.q_s, it.scale);
          __syncwarp();
          if (next < my_n) issue(next++);
        }
        if (ok) mma_to_gen(ms, gs, reinterpret_cast<float*>(sm.stage[warp][0]));
      } else {
        gen_init(gs);
        for (int j = 0; j < my_n; ++j) {
          const int st = acquire();
          if (st < 0) { ok = false; break; }
          ffma_group(reinterpret_cast<const char*>(sm.stage[warp][st]), gs, ptile,
                     qp_all + warp * kNH * kD, sm.q_s, it.scale);
          __syncwarp();
          if (next < my_n) issue(next++);
        }
      }
      if (!ok) {
        if (lane == 0) {
          report(a.status, S4KV_ERR_DEVICE_TIMEOUT, S4KV_DEV_TIMEOUT, item);
          atomicExch(&sm.abort_flag, 1);
        }
        while (consumed < issued) {   // let every copy in flight land before moving on
          const int st = consumed % kStages;
          mbar_wait(&sm.bar[warp][st], (consumed / kStages) & 1, kDrainNs);
          ++consumed;
        }
        gen_init(gs);
      } else {
        // tail: tokens past the last fully quantized group, 32 per chunk
        const int tail_lo = max(t_lo, t_main);
        for (int c0 = tail_lo + 32 * warp; c0 < t_hi; c0 += 32 * kWarps)
          generic_chunk(it, c0, min(32, t_hi - c0), gs, ptile, sm.q_s);
      }
    } else {
      gen_init(gs);
    }
    // per-warp state -> shared memory (the warp's own first stage buffer)
    {
      float* W = reinterpret_cast<float*>(sm.stage[warp][0]);   // M[8], L[8], O[8][128]
      if (lane == 0) {
#pragma unroll
        for (int hh = 0; hh < kNH; ++hh) {
          W[hh] = gs.m[hh];
          W[kNH + hh] = gs.l[hh];
        }
      }
#pragma unroll
      for (int hh = 0; hh < kNH; ++hh)
        *reinterpret_cast<float4*>(W + 2 * kNH + hh * kD + 4 * lane) =
            make_float4(gs.o[hh][0], gs.o[hh][1], gs.o[hh][2], gs.o[hh][3]);
    }
    __syncthreads();
    // merge the warps; write the output row or this item's partial
    float* ws_item = a.ws + static_cast<long long>(item) * a.g * (kD + 2);
    for (int i = tid; i < a.g * kD; i += kThreads) {
      const int j = i / kD, c = i % kD;
      float M = -INFINITY;
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, reinterpret_cast<const float*>(sm.stage[w][0])[j]);
      float O = 0.0f, L = 0.0f;
      if (M != -INFINITY) {
        for (int w = 0; w < kWarps; ++w) {
          const float* W = reinterpret_cast<const float*>(sm.stage[w][0]);
          const float al = exp2_safe(W[j] - M);
          O = fmaf(al, W[2 * kNH + j * kD + c], O);
          L = fmaf(al, W[kNH + j], L);
        }
      }
      if (direct) {
        const float y = L > 0.0f ? O / L : 0.0f;
        const long long o_idx = (static_cast<long long>(b) * a.Hq + h * a.g + j) * kD + c;
        if (a.out_dtype == S4KV_F32) reinterpret_cast<float*>(a.out)[o_idx] = y;
        else if (a.out_dtype == S4KV_F16) reinterpret_cast<__half*>(a.out)[o_idx] = __float2half_rn(y);
        else reinterpret_cast<__nv_bfloat16*>(a.out)[o_idx] = __float2bfloat16_rn(y);
      } else {
        ws_item[j * kD + c] = O;
        if (c == 0) {
          ws_item[a.g * kD + 2 * j] = M;
          ws_item[a.g * kD + 2 * j + 1] = L;
        }
      }
    }
    if (!direct) {
      __threadfence();
      __syncthreads();
      const int cslot = slot;
      if (tid == 0) {
        const int prev = atomicAdd(&a.counters[cslot * a.H + h], 1);
        sm.last = (prev == ns - 1);
      }
      __syncthreads();
      if (sm.last) {
        __threadfence();
        const float* base = a.ws + static_cast<long long>(pre[b] + h * ns) * a.g * (kD + 2);
        for (int i = tid; i < a.g * kD; i += kThreads) {
          const int j = i / kD, c = i % kD;
          float M = -INFINITY;
          for (int q = 0; q < ns; ++q)
            M = fmaxf(M, __ldcg(base + static_cast<long long>(q) * a.g * (kD + 2) + a.g * kD + 2 * j));
          float O = 0.0f, L = 0.0f;
          if (M != -INFINITY) {
            for (int q = 0; q < ns; ++q) {
              const float* P = base + static_cast<long long>(q) * a.g * (kD + 2);
              const float al = exp2_safe(__ldcg(P + a.g * kD + 2 * j) - M);
              O = fmaf(al, __ldcg(P + j * kD + c), O);
              L = fmaf(al, __ldcg(P + a.g * kD + 2 * j + 1), L);
            }
          }
          const float y = L > 0.0f ? O / L : 0.0f;
          const long long o_idx = (static_cast<long long>(b) * a.Hq + h * a.g + j) * kD + c;
          if (a.out_dtype == S4KV_F32) reinterpret_cast<float*>(a.out)[o_idx] = y;
          else if (a.out_dtype == S4KV_F16) reinterpret_cast<__half*>(a.out)[o_idx] = __float2half_rn(y);
          else reinterpret_cast<__nv_bfloat16*>(a.out)[o_idx] = __float2bfloat16_rn(y);
        }
        if (tid == 0) atomicExch(&a.counters[cslot * a.H + h], 0);
      }
    }
    __syncthreads();
  }
  // the last CTA out resets the work counter for the next launch
  if (tid == 0) {
    __threadfence();
    const int done = atomicAdd(a.work + 1, 1);
    if (done == static_cast<int>(gridDim.x) - 1) {
      atomicExch(a.work, 0);
      atomicExch(a.work + 1, 0);
    }
  }
}

}  // namespace

int decode_threads() { return kThreads; }

size_t decode_smem_bytes(int impl, int B) {
  const size_t base = impl == 1 ? prefix_offset<1>() : prefix_offset<0>();
  return base + static_cast<size_t>(B + 1) * sizeof(int);
}

namespace {
template <int IMPL>
cudaError_t prepare(int B, int* per_sm) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(decode_kernel<IMPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(decode_smem_bytes(IMPL, 8192)));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (per_sm)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, decode_kernel<IMPL>, kThreads,
                                                         decode_smem_bytes(IMPL, B));
  return cudaSuccess;
}
}  // namespace

int decode_ctas_per_sm(int impl, int B) {
  int n = 0;
  const cudaError_t e = impl == 0 ? prepare<0>(B, &n) : prepare<1>(B, &n);
  return e == cudaSuccess ? n : 0;
}

cudaError_t launch_decode(const DecodeArgs& a, int impl, int grid, cudaStream_t st) {
  const size_t smem = decode_smem_bytes(impl, a.B);
  cudaError_t e = impl == 0 ? prepare<0>(a.B, nullptr) : prepare<1>(a.B, nullptr);
  if (e != cudaSuccess) return e;
  if (impl == 0) decode_kernel<0><<<grid, kThreads, smem, st>>>(a);
  else decode_kernel<1><<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace s4kv
