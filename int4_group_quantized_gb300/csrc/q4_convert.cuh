// Conversion of one block of the decode copy of a weight (fg_pack_weight:
// 128 channels x 64 k, codes plus (scale, min) pairs) into the fp16 tensor-
// memory operand of a decode product (FlexGen notes, "5. 近似方法": weights
// stored in 4-bit groups of 64 along the output channel, converted back to
// FP16 before compute).
//
// Thread t of the warp that owns TMEM lane quarter q converts channels
// 32q + t/4 + 8w (w = 0..3) at the k pairs j = 4i + t%4 (i = 0..7): the
// register order of two 16x128b tensor-memory stores, a[16h + 2i + w'] being
// channel 32q + 16h + t/4 + 8w', column 4i + t%4 (two fp16 of consecutive k).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "fg.h"
#include "q4_dev.cuh"

namespace fg {
namespace q4 {

constexpr int kBlkCodes = 4096;   // code bytes of a block
__host__ __device__ constexpr int block_bytes(int fmt) {
  return kBlkCodes + (fmt == FG_PACK_EXACT ? 1024 : 512);   // 5120 or 4608
}

template <int FMT>
struct BlockConverter {
  uint4 w0, w1, pv[4];
  const uint8_t* blk;

  // Shared-memory loads of what this thread converts: its code words (the
  // fp16 pairs too, for FG_PACK_F16META; the fp32 pairs are read by convert).
  __device__ __forceinline__ void load(const uint8_t* block, int q, int lane) {
    blk = block;
    w0 = *reinterpret_cast<const uint4*>(block + q * 1024 + lane * 16);
    w1 = *reinterpret_cast<const uint4*>(block + q * 1024 + 512 + lane * 16);
    if (FMT == FG_PACK_F16META) {
      const uint4* pr = reinterpret_cast<const uint4*>(block + kBlkCodes + (q >> 1) * 256) + (lane & 3);
#pragma unroll
      for (int u = 0; u < 4; ++u) pv[u] = pr[4 * u];
    }
  }

  __device__ __forceinline__ void convert(uint32_t (&a)[32], int q, int lane) const {
    const int c4 = lane & 3;
    if (FMT == FG_PACK_EXACT) {
      // fp16(fmaf(q, scale, min)) with the stored fp32 pairs: the nibbles
      // become exact fp16 (1024 + q or 1024 + 16q, one lop3 for both k of a
      // pair), exact fp32 q by one mixed-precision op each, then one paired
      // fp32 FMA (each lane rounded once) and one rounding to fp16
      const float4* pr = reinterpret_cast<const float4*>(blk + kBlkCodes + (q >> 1) * 512) + c4;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 sm = pr[4 * i];   // (scale[2j], scale[2j+1], min[2j], min[2j+1]), j = 4i + c4
        const uint4 cw = i < 4 ? w0 : w1;
        const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
        const int e = i & 3;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t x = e >= 2 ? words[w] >> 8 : words[w];
          const uint32_t h = lop_mask_or(x, (e & 1) ? 0x00F000F0u : 0x000F000Fu, kMagic);
          const float2 qq = (e & 1) ? nib16_pair_f32(h) : nib_pair_f32(h);
          const float2 r = fma_f32x2(qq, make_float2(sm.x, sm.y), make_float2(sm.z, sm.w));
          a[16 * (w >> 1) + 2 * i + (w & 1)] = cvt_f16x2(r);
        }
      }
    } else {
      // fp16(q * scale' + min') in one fp16 FMA, (scale', min') the fp16 pairs
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 cw = u < 2 ? w0 : w1;
        const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          const int i = 2 * u + hi, e = i & 3;   // column 4i + c4: nibble slots e and e+4
          const uint32_t s2 = hi ? pv[u].z : pv[u].x, m2 = hi ? pv[u].w : pv[u].y;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint32_t x = e >= 2 ? words[w] >> 8 : words[w];
            a[16 * (w >> 1) + 2 * i + (w & 1)] =
                (e & 1) ? hfma2_u(hfma2_u(lop_mask_or(x, 0x00F000F0u, kMagic), kSixteenth, kNeg64), s2, m2)
                        : hfma2_u(hfma2_u(lop_mask_or(x, 0x000F000Fu, kMagic), kOne, kNegMagic), s2, m2);
          }
        }
      }
    }
  }
};

}  // namespace q4
}  // namespace fg
