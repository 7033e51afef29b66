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
  if (kmin == 0xffffffffu) {  // every member is NaN
    mn = mx = __uint_as_float(0x7fffffffu);
  } else {
    mn = key_to_float(kmin);
    mx = key_to_float(kmax);
  }
  const float r = __fsub_rn(mx, mn);
  // u = ((x - min) / r) * 15 with each op rounded as written decides the
  // code through rint.  One product t * (15 / r), with 15 / r rounded once
  // per group, is within 4 ulp of u (relative; u <= 15, so within 3.6e-6);
  // wherever it lies further than 1e-5 from a rounding boundary (k + 1/2)
  // both round to the same integer, and elsewhere -- or for a group whose r
  // is zero, infinite or NaN -- u itself is formed.  The codes equal those of
  // the literal op order.
  const float c15 = __fdiv_rn(15.0f, r);
  const bool fast = r > 0.0f && r < INFINITY && c15 < INFINITY;
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float t = __fsub_rn(v[i], mn);
    float u = __fmul_rn(t, c15);
    if (!fast || fabsf(fabsf(__fsub_rn(u, rintf(u))) - 0.5f) < 1e-5f) u = __fmul_rn(__fdiv_rn(t, r), 15.0f);
    const float q = fminf(fmaxf(rintf(u), 0.0f), 15.0f);  // NaN -> 0
    packed |= static_cast<uint32_t>(q) << (4 * i);
  }
  mn_out = mn;
  scale_out = __fdiv_rn(r, 15.0f);
  return packed;
}

}  // namespace codec
}  // namespace fg
