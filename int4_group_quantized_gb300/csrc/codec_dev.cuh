// Device-side group quantizer shared by the codec kernels and the fused
// KV append of the decode attention (FlexGen notes, "5. 近似方法",
// x_q = round((x - min)/(max - min) * 15) per group of 64).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace fg {
namespace codec {

// Monotone map from non-NaN floats to unsigned keys: a < b (with -0 < +0)
// iff key(a) < key(b).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// (min, max) of a group from the order keys of its non-NaN members; a group
// whose every member is NaN gets NaN for both.
__device__ __forceinline__ void group_bounds(uint32_t kmin, uint32_t kmax, float& mn, float& mx) {
  if (kmin == 0xffffffffu) {
    mn = mx = __uint_as_float(0x7fffffffu);
  } else {
    mn = key_to_float(kmin);
    mx = key_to_float(kmax);
  }
}

// The code of a member x of a group with minimum mn and range r = max - min
// is rint(((x - min) / r) * 15), each op rounded as written, clamped to
// [0, 15] (a NaN member gets 0).  code_exact forms exactly that.
__device__ __forceinline__ float code_exact(float x, float mn, float r) {
  const float u = __fmul_rn(__fdiv_rn(__fsub_rn(x, mn), r), 15.0f);
  return fminf(fmaxf(rintf(u), 0.0f), 15.0f);
}
// 1.5 * 2^23.  For u in [0, 2^22), u + kRound rounds u to the nearest
// integer, ties to even (the sum's ulp is 1), and holds that integer in its
// low mantissa bits; subtracting kRound again gives it as a float.  The
// rounding runs on the FMA pipe instead of the conversion unit.
constexpr float kRound = 12582912.0f;

// code_fast takes one product t * c15 with c15 = 15 / r rounded once per
// group (for r > 0 with r and c15 finite): it is within 4 ulp of the literal
// u (relative; u <= 15, so within 3.6e-6), so wherever it lies further than
// 1e-5 from a rounding boundary (k + 1/2) both round to the same integer.
// `near` is raised for a member closer than that; its code must then come
// from code_exact.  Returns kRound + code: here u <= 15 (1 + 2^-23), so the
// clamp to [0, 15] (NaN -> 0) before rounding changes no code and the
// boundary test may use the clamped code.
__device__ __forceinline__ float code_fast(float x, float mn, float c15, bool& near) {
  const float u = __fmul_rn(__fsub_rn(x, mn), c15);
  const float s = __fadd_rn(fminf(fmaxf(u, 0.0f), 15.0f), kRound);
  near |= fabsf(fabsf(__fsub_rn(u, __fsub_rn(s, kRound))) - 0.5f) < 1e-5f;
  return s;
}
__device__ __forceinline__ uint32_t code_bits(float s) { return __float_as_uint(s) & 15u; }
__device__ __forceinline__ bool code_is_near(float x, float mn, float c15) {
  bool near = false;
  code_fast(x, mn, c15, near);
  return near;
}

// Quantizes the 64-group held by 8 consecutive lanes {8j .. 8j+7} of a warp
// (lane 8j+p holds elements 8p .. 8p+7 in v).  Every lane of the warp must
// call it (the reduction uses full-warp shuffles).  Returns the lane's 8
// codes packed low nibble first; mn_out/scale_out are valid on all 8 lanes.
// Each operation is an explicitly rounded fp32 intrinsic: no contraction.
__device__ __forceinline__ uint32_t quantize_group8(const float (&v)[8], float& mn_out,
                                                   float& scale_out) {
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (!isnan(v[i])) {
      const uint32_t k = order_key(v[i]);
      kmin = min(kmin, k);
      kmax = max(kmax, k);
    }
  }
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, off));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, off));
  }
  float mn, mx;
  group_bounds(kmin, kmax, mn, mx);
  const float r = __fsub_rn(mx, mn);
  const float c15 = __fdiv_rn(15.0f, r);
  const bool fast = r > 0.0f && r < INFINITY && c15 < INFINITY;
  uint32_t q[8];
  bool near = false;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    q[i] = fast ? code_bits(code_fast(v[i], mn, c15, near)) : static_cast<uint32_t>(code_exact(v[i], mn, r));
  if (near) {   // rare: a member within 1e-5 of a rounding boundary
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (code_is_near(v[i], mn, c15)) q[i] = static_cast<uint32_t>(code_exact(v[i], mn, r));
  }
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) packed |= q[i] << (4 * i);
  mn_out = mn;
  scale_out = __fdiv_rn(r, 15.0f);
  return packed;
}

// A code as a float, exactly (q in 0..15): the round-by-addition in reverse.
__device__ __forceinline__ float code_float(uint32_t q) { return __fsub_rn(__uint_as_float(0x4B400000u | q), kRound); }

}  // namespace codec
}  // namespace fg
