// Device helpers that turn 4-bit weight codes into fp16 operands for the
// tensor cores (FlexGen notes, "5. 近似方法": weights stored in 4-bit groups,
// converted back to FP16 before compute).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace fg {
namespace q4 {

__device__ __forceinline__ uint32_t lop_mask_or(uint32_t x, uint32_t mask, uint32_t magic) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "r"(mask), "r"(magic));  // (x & mask) | magic
  return r;
}
__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t bcast_h2(float v) {
  const __half2 h = __float2half2_rn(v);
  return *reinterpret_cast<const uint32_t*>(&h);
}

constexpr uint32_t kMagic = 0x64006400u;      // fp16 (1024, 1024)
constexpr uint32_t kNegMagic = 0xE400E400u;   // fp16 (-1024, -1024)
constexpr uint32_t kOne = 0x3C003C00u;        // fp16 (1, 1)
constexpr uint32_t kSixteenth = 0x2C002C00u;  // fp16 (1/16, 1/16)
constexpr uint32_t kNeg64 = 0xD400D400u;      // fp16 (-64, -64)

// fp16x2 h = (1024 + q0, 1024 + q1), q0, q1 in 0..15 -> exact fp32 (q0, q1),
// one mixed-precision add per half.
__device__ __forceinline__ float2 nib_pair_f32(uint32_t h) {
  float lo, hi;
  asm("{ .reg .f16 a, b; mov.b32 {a, b}, %2; add.rn.f32.f16 %0, a, %3; add.rn.f32.f16 %1, b, %3; }"
      : "=f"(lo), "=f"(hi)
      : "r"(h), "f"(-1024.0f));
  return make_float2(lo, hi);
}
// fp16x2 h = (1024 + 16 q0, 1024 + 16 q1) -> exact fp32 (q0, q1): h/16 - 64
// in one mixed-precision fma per half (both steps exact).
__device__ __forceinline__ float2 nib16_pair_f32(uint32_t h) {
  float lo, hi;
  asm("{ .reg .f16 a, b, c; mov.b32 {a, b}, %2; mov.b16 c, 0x2C00; fma.rn.f32.f16 %0, a, c, %3; "
      "fma.rn.f32.f16 %1, b, c, %3; }"
      : "=f"(lo), "=f"(hi)
      : "r"(h), "f"(-64.0f));
  return make_float2(lo, hi);
}
// Two IEEE fp32 fmas (each rounded once, round to nearest even) in one
// paired instruction: (a.x * b.x + c.x, a.y * b.y + c.y).
__device__ __forceinline__ float2 fma_f32x2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{ .reg .b64 ra, rb, rc, rd; mov.b64 ra, {%2, %3}; mov.b64 rb, {%4, %5}; mov.b64 rc, {%6, %7};\n"
      "fma.rn.f32x2 rd, ra, rb, rc; mov.b64 {%0, %1}, rd; }"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
// fp16x2 (round to nearest even) of (v.x, v.y): v.x in the lower half.
__device__ __forceinline__ uint32_t cvt_f16x2(float2 v) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(v.y), "f"(v.x));
  return r;
}

// 8 codes (one 32-bit word: consecutive output channels n..n+7 of one input
// row, one 64-group) -> 8 fp16 weights q*scale + min (s2, m2: scale and min
// broadcast to both fp16 halves).  A lop3 with the fp16 exponent of 1024
// turns nibble c into the exact value 1024 + c (or 1024 + 16c for the upper
// nibble of a byte); one fp16x2 FMA removes the offset exactly, a second
// applies (scale, min).  The pairs come out as channels (0,4) (1,5) (2,6)
// (3,7); a 16-byte chunk keeps that order (see perm8).
__device__ __forceinline__ uint4 dequant8(uint32_t c, uint32_t s2, uint32_t m2) {
  const uint32_t y = c >> 8;
  const uint32_t t0 = hfma2_u(lop_mask_or(c, 0x000F000Fu, kMagic), kOne, kNegMagic);     // (c0, c4)
  const uint32_t t1 = hfma2_u(lop_mask_or(c, 0x00F000F0u, kMagic), kSixteenth, kNeg64);  // (c1, c5)
  const uint32_t t2 = hfma2_u(lop_mask_or(y, 0x000F000Fu, kMagic), kOne, kNegMagic);     // (c2, c6)
  const uint32_t t3 = hfma2_u(lop_mask_or(y, 0x00F000F0u, kMagic), kSixteenth, kNeg64);  // (c3, c7)
  return make_uint4(hfma2_u(t0, s2, m2), hfma2_u(t1, s2, m2), hfma2_u(t2, s2, m2), hfma2_u(t3, s2, m2));
}

// Position p (0..7) of a dequant8 chunk holds channel perm8(p) of its 8.
__device__ __forceinline__ int perm8(int p) { return ((p & 1) << 2) | (p >> 1); }

}  // namespace q4
}  // namespace fg
