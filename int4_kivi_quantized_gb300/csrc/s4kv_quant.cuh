// Warp-level write side of the cache, shared by the append kernels and the
// fused decode step: the exact quantizer, one value token into its page
// record, one key group into its two page records, one FP8 token.
//
// Method ("4.4 KV Cache 量化", sections 3.1 and 3.2): a key group is G = 32
// consecutive tokens of one channel, a value group Gv = 32 channels of one
// token; each keeps fp32 (scale, min) and codes of the min/max asymmetric
// mapping. Every rounding is an explicit IEEE intrinsic (__fsub_rn, __fdiv_rn,
// __float2int_rn, __fadd_rn), so no compiler contraction can change a code.
#pragma once

#include "s4kv_common.cuh"

#include <cuda_fp8.h>

namespace s4kv {
namespace quant {

// Code of x for a group with minimum lo and scale s: rne((x - lo) / s) with
// each step one binary32 rounding, clamped to 0 .. 2^BITS - 1; s == 0 gives 0.
template <int BITS>
__device__ __forceinline__ int code(float x, float lo, float s) {
  if (s == 0.0f) return 0;
  const int c = __float2int_rn(__fdiv_rn(__fsub_rn(x, lo), s));
  return min(max(c, 0), Rec<BITS>::kLevels);
}

// The same code through the correctly rounded reciprocal r = fl(1 / s) (0 when
// s is 0 or below kMinFastScale): t' = fl(fl(x - lo) * r) is within 2^-19 of the
// quotient for codes below 16 and fl(quotient) within 2^-21 of it, so when t' is
// farther than 2^-17 from every half-integer it rounds to the division's code;
// otherwise (and without r) the division decides.
constexpr float kMinFastScale = 7.8886091e-31f;   // 2^-100
constexpr float kTieGuard = 0.4999923706054688f;  // 0.5 - 2^-17
template <int BITS>
__device__ __forceinline__ int code_fast(float x, float lo, float s, float r) {
  if (r == 0.0f) return code<BITS>(x, lo, s);
  const float t = __fmul_rn(__fsub_rn(x, lo), r);
  const float f = __fsub_rn(__fadd_rn(t, 12582912.0f), 12582912.0f);   // rne(t): 1.5 * 2^23
  if (!(fabsf(__fsub_rn(t, f)) <= kTieGuard)) return code<BITS>(x, lo, s);
  return min(max(static_cast<int>(f), 0), Rec<BITS>::kLevels);
}

// Record bytes of one value token (absolute position t) from this lane's four
// values raw (channels 4l .. 4l+3, 16-bit), by one warp: the 8 lanes of a
// 32-channel group reduce min and max by shuffles. rec: the token's page record
// of this kv head, or null (nothing is written; every lane must still call).
template <int BITS>
__device__ __forceinline__ void value_token(char* rec, int t, uint2 raw, int dtype) {
  using F = Rec<BITS>;
  const int l = threadIdx.x & 31;
  float x[4];
  x[0] = widen16(static_cast<uint16_t>(raw.x & 0xffff), dtype);
  x[1] = widen16(static_cast<uint16_t>(raw.x >> 16), dtype);
  x[2] = widen16(static_cast<uint16_t>(raw.y & 0xffff), dtype);
  x[3] = widen16(static_cast<uint16_t>(raw.y >> 16), dtype);
  float lo = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
  float hi = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, m));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, m));
  }
  lo = __fadd_rn(lo, 0.0f);   // -0 becomes +0
  hi = __fadd_rn(hi, 0.0f);
  const float s = __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(F::kLevels));
  // codes through the reciprocal (see code_fast), the division where it decides
  const float rs = s >= kMinFastScale ? __frcp_rn(s) : 0.0f;
  int c4 = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) c4 |= code_fast<BITS>(x[q], lo, s, rs) << (4 * q);
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
  if (!rec) return;
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

__device__ __forceinline__ uint32_t bytes_0213(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b2, 0x0040), __byte_perm(b1, b3, 0x0040), 0x5410);
}

// Key codes and key metadata of one complete key group, by one warp: rows[t]
// (t = 0..31, this lane's channels 4l .. 4l+3 as four 16-bit values) are the
// group's tokens; rec0 and rec1 are the records of its two pages for this kv
// head (either may be null: that page is skipped). Lane l owns the channels
// 32b + 4kk + j with b = l / 8, kk = l % 8: exactly the channels of record word
// (kk, L = 4a + b), so it writes its words whole.
template <int BITS>
__device__ __forceinline__ void key_group(char* rec0, char* rec1, const uint2 (&rows)[kG], int dtype) {
  using F = Rec<BITS>;
  const int l = threadIdx.x & 31;
  const int kk = l & 7, b = l >> 3;
  float lo[4], s[4], rs[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float mn = INFINITY, mx = -INFINITY;
#pragma unroll
    for (int t = 0; t < kG; ++t) {
      const uint32_t w = j < 2 ? rows[t].x : rows[t].y;
      const float v = widen16(static_cast<uint16_t>((j & 1) ? (w >> 16) : (w & 0xffff)), dtype);
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
    }
    lo[j] = __fadd_rn(mn, 0.0f);
    const float hi = __fadd_rn(mx, 0.0f);
    s[j] = __fdiv_rn(__fsub_rn(hi, lo[j]), static_cast<float>(F::kLevels));
    rs[j] = s[j] >= kMinFastScale ? __frcp_rn(s[j]) : 0.0f;
  }
  auto cd = [&](int t, int j) -> uint32_t {
    const uint32_t w = j < 2 ? rows[t].x : rows[t].y;
    const float v = widen16(static_cast<uint16_t>((j & 1) ? (w >> 16) : (w & 0xffff)), dtype);
    return static_cast<uint32_t>(code_fast<BITS>(v, lo[j], s[j], rs[j]));
  };
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    char* rec = p ? rec1 : rec0;
#pragma unroll
    for (int a = 0; a < 8; ++a) {
      const int t0 = 16 * p + a;
      if constexpr (BITS == 4) {
        const uint32_t w = bytes_0213(cd(t0, 0) | (cd(t0 + 8, 0) << 4), cd(t0, 1) | (cd(t0 + 8, 1) << 4),
                                      cd(t0, 2) | (cd(t0 + 8, 2) << 4), cd(t0, 3) | (cd(t0 + 8, 3) << 4));
        if (rec) *reinterpret_cast<uint32_t*>(rec + F::kKc + (kk >> 2) * 512 + (4 * a + b) * 16 + (kk & 3) * 4) = w;
      } else {
        // positions 0, 1 (token a, a + 8) of slice kk; slice kk + 1 (lane l + 1)
        // brings positions 2, 3
        uint32_t B[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t mine = cd(t0, j) | (cd(t0 + 8, j) << 2);
          const uint32_t other = __shfl_down_sync(0xffffffffu, mine, 1);
          B[j] = mine | (other << 4);
        }
        if (rec && (kk & 1) == 0)
          *reinterpret_cast<uint32_t*>(rec + F::kKc + (4 * a + b) * 16 + (kk >> 1) * 4) = bytes_0213(B[0], B[1], B[2], B[3]);
      }
    }
  }
  // metadata: channel 64 j + 32 u + 4 i + e lives in page j at 16 (2i + u) + 4e
  {
    char* rec = (l >> 4) ? rec1 : rec0;
    const int u = (l >> 3) & 1, i = l & 7;
    if (rec) {
      *reinterpret_cast<float4*>(rec + F::kKm + (2 * i + u) * 16) = make_float4(s[0], s[1], s[2], s[3]);
      *reinterpret_cast<float4*>(rec + F::kKm + (2 * i + u) * 16 + 256) = make_float4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
}

// One new token (position t within its page record rec) of FP8 E4M3 pages, by
// one warp: lane l converts channels 4l .. 4l+3 of its key and value rows (the
// division by the head's scale rounded to fp32, then the saturating
// round-to-nearest-even E4M3 conversion) and stores them in place.
__device__ __forceinline__ uint32_t e4m3_of(float x, float scale) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fdiv_rn(x, scale), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ void fp8_token(char* rec, int t, uint2 kr, uint2 vr, float ks, float vs, int dtype) {
  const int lane = threadIdx.x & 31;
  const int tau = t % kP;
  const uint16_t kx[4] = {static_cast<uint16_t>(kr.x & 0xffff), static_cast<uint16_t>(kr.x >> 16),
                          static_cast<uint16_t>(kr.y & 0xffff), static_cast<uint16_t>(kr.y >> 16)};
  const uint16_t vx[4] = {static_cast<uint16_t>(vr.x & 0xffff), static_cast<uint16_t>(vr.x >> 16),
                          static_cast<uint16_t>(vr.y & 0xffff), static_cast<uint16_t>(vr.y >> 16)};
  uint32_t kc[4], vc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    kc[q] = e4m3_of(widen16(kx[q], dtype), ks);
    vc[q] = e4m3_of(widen16(vx[q], dtype), vs);
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

}  // namespace quant
}  // namespace s4kv
