// Activations for the MXFP4 expert path: every bf16 token row (x before the gate/up pass, h
// before the down pass) is carried as two E4M3 terms with E8M0 scales, one scale byte per 32
// consecutive elements and term:
//     v = hi * 2^(a - 127) + lo * 2^(b - 127) + e.
// a puts the block's largest |v| in [128, 256) and hi is v / 2^(a-127) rounded to nearest E4M3;
// b does the same for the remainders r = v - hi * 2^(a-127), and lo is r / 2^(b-127) rounded.
// With a largest |r| of at most 8 * 2^(a-127) (half an E4M3 step at 128..256), |e| is at most
// half a step of lo at its largest, 8 * 2^(b-127) <= 2^-8 of the block's largest |v|: about the
// rounding of that largest element to bf16.
//
// The tensor core's block-scaled MMA (kind::mxf8f6f4) applies the scales, so a product with an
// MXFP4 weight row is (hi + lo terms) exactly as written above, accumulated in fp32.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {
namespace mx {

// Layout of one encoded [rows, K] activation matrix in the workspace: the hi and lo code planes
// ([rows, K] bytes each, 16-byte aligned for TMA) and their scale planes ([rows, K/32] bytes).
struct Planes {
  uint8_t* hi;
  uint8_t* lo;
  uint8_t* s_hi;
  uint8_t* s_lo;
};

inline Planes planes_at(char* base, long rows, long K) {
  Planes p;
  p.hi = reinterpret_cast<uint8_t*>(base);
  p.lo = p.hi + rows * K;
  p.s_hi = p.lo + rows * K;
  p.s_lo = p.s_hi + rows * (K / 32);
  return p;
}

inline size_t planes_bytes(long rows, long K) { return (size_t)rows * (2 * K + 2 * (K / 32)); }

// Scale byte of a block with largest magnitude amax: 2^(a-127) maps amax into [128, 256).
__device__ __forceinline__ uint32_t scale_byte(float amax) {
  if (!(amax > 0.f)) return 127u;
  const int E = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
  return (uint32_t)min(max(E - 7, 1), 253);
}

// 2^(127 - a) and 2^(a - 127) for a in [1, 253] (both normal fp32).
__device__ __forceinline__ float inv_scale(uint32_t a) { return __uint_as_float((254u - a) << 23); }
__device__ __forceinline__ float scale_value(uint32_t a) { return __uint_as_float(a << 23); }

// Two fp32 values -> two E4M3 codes (lo in bits 0..7), round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes (bits 0..15 of `two`) -> their exact values.
__device__ __forceinline__ float2 e4m3x2_value(uint32_t two) {
  uint32_t h;
  asm("{\n"
      "  .reg .b16 c;\n"
      "  cvt.u16.u32 c, %1;\n"
      "  cvt.rn.f16x2.e4m3x2 %0, c;\n"
      "}"
      : "=r"(h)
      : "r"(two));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One thread, one block of 32 values: the hi and lo code bytes (4 words each, element 4i+j in
// byte j of word i) and the two scale bytes.
__device__ __forceinline__ void encode32(const float (&v)[32], uint32_t (&hi)[8], uint32_t (&lo)[8],
                                         uint32_t& a, uint32_t& b) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  a = scale_byte(amax);
  const float ia = inv_scale(a), sa = scale_value(a);
  float r[32];
  float rmax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const uint32_t c = e4m3x2(v[i] * ia, v[i + 1] * ia);
    const float2 q = e4m3x2_value(c);
    r[i] = v[i] - q.x * sa;
    r[i + 1] = v[i + 1] - q.y * sa;
    rmax = fmaxf(rmax, fmaxf(fabsf(r[i]), fabsf(r[i + 1])));
    if ((i & 2) == 0) hi[i >> 2] = c;
    else hi[i >> 2] |= c << 16;
  }
  b = scale_byte(rmax);
  const float ib = inv_scale(b);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const uint32_t c = e4m3x2(r[i] * ib, r[i + 1] * ib);
    if ((i & 2) == 0) lo[i >> 2] = c;
    else lo[i >> 2] |= c << 16;
  }
}

// One warp, one block of 32 values (lane i holds element i), for two blocks at once (v0 and
// v1): each lane gets its own hi and lo bytes; every lane gets the scale bytes.
__device__ __forceinline__ void encode_warp2(float v0, float v1, uint32_t& hi0, uint32_t& lo0,
                                             uint32_t& hi1, uint32_t& lo1, uint32_t& a0,
                                             uint32_t& b0, uint32_t& a1, uint32_t& b1) {
  float m0 = fabsf(v0), m1 = fabsf(v1);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
  }
  a0 = scale_byte(m0);
  a1 = scale_byte(m1);
  const uint32_t c = e4m3x2(v0 * inv_scale(a0), v1 * inv_scale(a1));
  const float2 q = e4m3x2_value(c);
  const float r0 = v0 - q.x * scale_value(a0), r1 = v1 - q.y * scale_value(a1);
  hi0 = c & 0xFFu;
  hi1 = (c >> 8) & 0xFFu;
  float n0 = fabsf(r0), n1 = fabsf(r1);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    n0 = fmaxf(n0, __shfl_xor_sync(0xffffffffu, n0, o));
    n1 = fmaxf(n1, __shfl_xor_sync(0xffffffffu, n1, o));
  }
  b0 = scale_byte(n0);
  b1 = scale_byte(n1);
  const uint32_t l = e4m3x2(r0 * inv_scale(b0), r1 * inv_scale(b1));
  lo0 = l & 0xFFu;
  lo1 = (l >> 8) & 0xFFu;
}

}  // namespace mx
}  // namespace moe
