// Device helpers shared by the decode-attention kernels (dense and top-K):
// the launch arguments, the warp-level MMA on biased integer codes, q as MMA
// B fragments, and the Concat of the new token into the 4-bit cache
// (FlexGen notes, "背景知识" decode equations; "5. 近似方法": K/V stored in
// 4-bit groups of 64 along the hidden dimension).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "codec_dev.cuh"

namespace fg {
namespace attn {

struct DecodeArgs {
  uint8_t* kc;   // codes [b*H][cap][D/2]
  uint8_t* vc;
  float* kmin;   // [b*H][cap][D/64]
  float* kscale;
  float* vmin;
  float* vscale;
  const __half* q;     // row bi at q + bi*ldq, head h at + h*D
  int64_t ldq;
  const __half* knew;  // new token's K/V rows (nullptr: nothing to append)
  const __half* vnew;
  int64_t ldnew;
  int64_t pos;         // slot of the new token; attend over 0..pos
  __half* out;         // [b][ldo]
  int64_t ldo;
  float* part;         // splits > 1: [b*H][splits][D + 2]
  int heads;
  int64_t cap;
  int splits;
  int tps;             // tokens per split (multiple of 16)
  unsigned int* err;   // device error word (bounded waits of the staged kernels)
  uint32_t wait_limit; // polls of a bounded wait
};

__device__ __forceinline__ uint32_t lop_mask_or(uint32_t x, uint32_t mask, uint32_t magic) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "r"(mask), "r"(magic));  // (x & mask) | magic
  return r;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_h2(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

constexpr uint32_t kMagic = 0x64006400u;   // fp16 1024.0 in both halves
constexpr uint32_t kLoNib = 0x000F000Fu;   // nibble 0 of bytes 0 and 2
constexpr uint32_t kHiNib = 0x00F000F0u;   // nibble 1 of bytes 0 and 2 (value x16)

// Concat: warp 0 quantizes the new token's K and V rows into slot pos
// (8 lanes per 64-group, the codec's rounding).
template <int D>
__device__ __forceinline__ void append_token(const DecodeArgs& a, int64_t slot0, int64_t bi, int h, int lane) {
  constexpr int NG = D / 64;
  const int gi = lane >> 3, part = lane & 7;
  const bool valid = gi < 2 * NG;
  const int which = gi / NG, grp = gi % NG;
  float v[8];
  if (valid) {
    const __half* src = (which ? a.vnew : a.knew) + bi * a.ldnew + h * D + grp * 64 + part * 8;
    const uint4 raw = *reinterpret_cast<const uint4*>(src);
    const __half2* hh = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(hh[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.0f;
  }
  float mn, sc;
  const uint32_t packed = codec::quantize_group8(v, mn, sc);
  if (valid) {
    const int64_t slot = slot0 + a.pos;
    *reinterpret_cast<uint32_t*>((which ? a.vc : a.kc) + slot * (D / 2) + grp * 32 + part * 4) = packed;
    if (part == 0) {
      (which ? a.vmin : a.kmin)[slot * NG + grp] = mn;
      (which ? a.vscale : a.kscale)[slot * NG + grp] = sc;
    }
  }
}

// q of one (sequence, head) as this lane's B fragments: lane (gq, tig)
// supplies k-indices {2tig, 2tig+1, 2tig+8, 2tig+9} of every k-step; they
// stand for its own dims: per group, dims 16*tig .. 16*tig+15, taken from two
// 32-bit code words as (0,4),(1,5)x16 | (2,6),(3,7)x16.
template <int D, class S>
__device__ __forceinline__ void setup_q(S& W, const __half* qrow, int tig) {
  constexpr int NG = D / 64;
  auto& qb = W.qb;
  auto& bias = W.bias;
  auto& qsum = W.qsum;
  {
    // q stays exact (it is fp16 already); log2(e)/sqrt(d) is applied to the
    // fp32 scores instead, so no rounding of a scaled q enters them
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      float qv[16];
      const uint4* src = reinterpret_cast<const uint4*>(qrow + g * 64 + 16 * tig);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint4 raw = src[c];
        const __half2* hh = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(hh[i]);
          qv[8 * c + 2 * i] = f.x;
          qv[8 * c + 2 * i + 1] = f.y;
        }
      }
      float bsum = 0.0f, qs = 0.0f;
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const float* d = qv + 8 * w;
        qb[g][2 * w][0] = pack_h2(d[0], d[4]);
        qb[g][2 * w][1] = pack_h2(d[1] * 0.0625f, d[5] * 0.0625f);
        qb[g][2 * w + 1][0] = pack_h2(d[2], d[6]);
        qb[g][2 * w + 1][1] = pack_h2(d[3] * 0.0625f, d[7] * 0.0625f);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const float2 x = unpack_h2(qb[g][2 * w + s][0]);
          const float2 y = unpack_h2(qb[g][2 * w + s][1]);
          bsum += x.x + x.y + y.x + y.y;
          qs += x.x + x.y + 16.0f * (y.x + y.y);
        }
      }
      bsum += __shfl_xor_sync(0xffffffffu, bsum, 1);
      bsum += __shfl_xor_sync(0xffffffffu, bsum, 2);
      qs += __shfl_xor_sync(0xffffffffu, qs, 1);
      qs += __shfl_xor_sync(0xffffffffu, qs, 2);
      bias[g] = 1024.0f * bsum;
      qsum[g] = qs;
    }
  }
}

// Scores of tokens gq and gq+8 of a 16-token block (rows gq and gq+8 of this
// lane's m16n8k16 fragments; every lane of a row ends with the full sum),
// before the softmax scale: per 64-group, scale * (sum_j q_j c_j) + min *
// (sum_j q_j).  Q holds q as B fragments (setup_q); kw are the two rows'
// codes (8 bytes per group at dims 16*tig of the group), ksc/kmn their
// (scale, min) pairs.
template <int NG, class S>
__device__ __forceinline__ void block_scores(const S& Q, const uint2 (&kw)[2][NG], const float (&ksc)[2][NG],
                                             const float (&kmn)[2][NG], float& sc0, float& sc1) {
  sc0 = 0.0f;
  sc1 = 0.0f;
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const uint32_t x0 = w ? kw[0][g].y : kw[0][g].x;
      const uint32_t x1 = w ? kw[1][g].y : kw[1][g].x;
      mma16816(d, lop_mask_or(x0, kLoNib, kMagic), lop_mask_or(x1, kLoNib, kMagic),
               lop_mask_or(x0, kHiNib, kMagic), lop_mask_or(x1, kHiNib, kMagic), Q.qb[g][2 * w][0],
               Q.qb[g][2 * w][1]);
      const uint32_t y0 = x0 >> 8, y1 = x1 >> 8;
      mma16816(d, lop_mask_or(y0, kLoNib, kMagic), lop_mask_or(y1, kLoNib, kMagic),
               lop_mask_or(y0, kHiNib, kMagic), lop_mask_or(y1, kHiNib, kMagic), Q.qb[g][2 * w + 1][0],
               Q.qb[g][2 * w + 1][1]);
    }
    sc0 += ksc[0][g] * (d[0] - Q.bias[g]) + kmn[0][g] * Q.qsum[g];
    sc1 += ksc[1][g] * (d[2] - Q.bias[g]) + kmn[1][g] * Q.qsum[g];
  }
}

// log2(e)/sqrt(d): the fp32 scores are scaled once into base 2 for exp2
template <int D>
__device__ __forceinline__ constexpr float score_scale_log2() {
  return static_cast<float>(1.4426950408889634074 * (D == 128 ? 0.088388347648318440550 : 0.125));
}

}  // namespace attn
}  // namespace fg
