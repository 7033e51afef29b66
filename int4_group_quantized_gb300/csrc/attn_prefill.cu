// Causal prefill attention over the 4-bit KV cache on the tensor cores
// (FlexGen notes, "背景知识": x_Out = Softmax(x_Q x_K^T / sqrt(h1)) x_V with a
// causal mask for generation; "5. 近似方法": K/V stored in 4-bit groups of 64
// along the hidden dimension and converted back to FP16 before compute).
//
// Flash-style: one CTA (4 warps) per (sequence, head, 64 queries); each warp
// owns 16 query rows.  Keys are walked 64 at a time: the CTA converts the
// chunk's K and V codes to fp16 in shared memory (fmaf(q, scale, min) in
// fp32, rounded to fp16 -- the same values the codec's dequantization gives),
// then every warp forms S = Q K^T with m16n8k16 MMAs (fp32 accumulate), keeps
// a running max and sum in base 2 (scores scaled by log2(e)/sqrt(d) in fp32),
// re-uses the S accumulators as the A operand of P V, and rescales its output
// accumulators when the max moves.  Chunks wholly above a warp's rows are
// skipped; the diagonal chunk is masked.
#include <math.h>

#include "fg_internal.cuh"

namespace fg {
namespace {

constexpr int QB = 64;    // queries per CTA
constexpr int KC = 64;    // keys per chunk

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

struct PrefillArgs {
  const uint32_t* kc;   // codes as words, [b*H][cap][D/8]
  const uint32_t* vc;
  const float* kmin;    // [b*H][cap][D/64]
  const float* kscale;
  const float* vmin;
  const float* vscale;
  const __half* q;      // row (bi*s + t) at q + row*ldq, head h at + h*D
  int64_t ldq;
  __half* out;          // same layout, ldo
  int64_t ldo;
  int64_t s;
  int heads;
  int64_t cap;
};

template <int D>
__global__ void __launch_bounds__(128) prefill_attn_mma_kernel(const PrefillArgs a) {
  constexpr int NKS = D / 16;   // k-steps of Q K^T
  constexpr int NDT = D / 8;    // n8 tiles of output dims
  constexpr int NG = D / 64;
  constexpr int LD = D + 8;     // padded rows: ldmatrix rows hit distinct banks
  __shared__ __align__(16) __half Ks[KC][LD];
  __shared__ __align__(16) __half Vs[KC][LD];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int64_t nqb = (a.s + QB - 1) / QB;
  const int64_t qb = blockIdx.x % nqb, bh = blockIdx.x / nqb;
  const int64_t bi = bh / a.heads;
  const int h = static_cast<int>(bh % a.heads);
  const int64_t q0 = qb * QB;
  const int64_t wr0 = q0 + warp * 16;                 // first query row of this warp
  const int64_t kend = min(q0 + QB, a.s);             // keys the CTA needs: 0..kend-1
  const int64_t slot0 = bh * a.cap;

  // Q as A fragments, exact (fp16 already); log2(e)/sqrt(d) is applied to
  // the fp32 scores, so that no rounding of a scaled Q enters them
  constexpr float kQs = static_cast<float>(1.4426950408889634074 * (D == 128 ? 0.088388347648318440550 : 0.125));
  uint32_t qa[NKS][4];
  {
    const int64_t r0 = wr0 + g, r1 = wr0 + g + 8;
#pragma unroll
    for (int kk = 0; kk < NKS; ++kk) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t r = (e & 1) ? r1 : r0;
        const int c = 16 * kk + 2 * tig + 8 * (e >> 1);
        float2 f = make_float2(0.0f, 0.0f);
        if (r < a.s) f = __half22float2(*reinterpret_cast<const __half2*>(a.q + (bi * a.s + r) * a.ldq + h * D + c));
        qa[kk][e] = pack_h2(f.x, f.y);
      }
    }
  }

  float oacc[NDT][4];
#pragma unroll
  for (int i = 0; i < NDT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
  const int mi = lane >> 3, ri = lane & 7;

  for (int64_t kc = 0; kc < kend; kc += KC) {
    __syncthreads();   // the previous chunk is no longer read
    for (int i = threadIdx.x; i < 2 * KC * (D / 8); i += 128) {
      const int which = i / (KC * (D / 8));
      const int r = (i / (D / 8)) % KC, w = i % (D / 8);
      const int64_t key = kc + r;
      uint4 o = make_uint4(0u, 0u, 0u, 0u);
      if (key < kend) {
        const int64_t slot = slot0 + key;
        const uint32_t c = (which ? a.vc : a.kc)[slot * (D / 8) + w];
        const float mn = (which ? a.vmin : a.kmin)[slot * NG + (w >> 3)];
        const float sc = (which ? a.vscale : a.kscale)[slot * NG + (w >> 3)];
        uint32_t* ov = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          ov[j] = pack_h2(__fmaf_rn(static_cast<float>((c >> (8 * j)) & 15u), sc, mn),
                          __fmaf_rn(static_cast<float>((c >> (8 * j + 4)) & 15u), sc, mn));
      }
      *reinterpret_cast<uint4*>(&(which ? Vs : Ks)[r][w * 8]) = o;
    }
    __syncthreads();
    if (wr0 >= a.s || kc > wr0 + 15) continue;        // no row of this warp sees these keys

    // S = Q K^T for 16 rows x 64 keys
    float sacc[KC / 8][4];
#pragma unroll
    for (int i = 0; i < KC / 8; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < NKS; ++kk) {
#pragma unroll
      for (int nt = 0; nt < KC / 8; nt += 2) {
        uint32_t r[4];
        ldsm_x4(r, &Ks[8 * nt + 8 * (mi >> 1) + ri][16 * kk + 8 * (mi & 1)]);
        mma16816(sacc[nt], qa[kk], r[0], r[1]);
        mma16816(sacc[nt + 1], qa[kk], r[2], r[3]);
      }
    }
#pragma unroll
    for (int i = 0; i < KC / 8; ++i) {
      sacc[i][0] *= kQs;
      sacc[i][1] *= kQs;
      sacc[i][2] *= kQs;
      sacc[i][3] *= kQs;
    }
    // causal mask and sequence end (only where the chunk reaches them)
    if (kc + KC > wr0 || kc + KC > a.s) {
#pragma unroll
      for (int nt = 0; nt < KC / 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t key = kc + 8 * nt + 2 * tig + (e & 1);
          const int64_t row = wr0 + g + 8 * (e >> 1);
          if (key > row || key >= kend) sacc[nt][e] = -INFINITY;
        }
      }
    }
    // online softmax, base 2
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < KC / 8; ++nt) {
      mx0 = fmaxf(mx0, fmaxf(sacc[nt][0], sacc[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(sacc[nt][2], sacc[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);   // finite: key kc <= row for every live row
    const float al0 = exp2f(m0 - n0), al1 = exp2f(m1 - n1);
    m0 = n0;
    m1 = n1;
    l0 *= al0;
    l1 *= al1;
#pragma unroll
    for (int i = 0; i < NDT; ++i) {
      oacc[i][0] *= al0;
      oacc[i][1] *= al0;
      oacc[i][2] *= al1;
      oacc[i][3] *= al1;
    }
    uint32_t pa[KC / 16][4];
#pragma unroll
    for (int nt = 0; nt < KC / 8; ++nt) {
      const float p0 = exp2f(sacc[nt][0] - n0), p1 = exp2f(sacc[nt][1] - n0);
      const float p2 = exp2f(sacc[nt][2] - n1), p3 = exp2f(sacc[nt][3] - n1);
      l0 += p0 + p1;
      l1 += p2 + p3;
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack_h2(p0, p1);   // row g,   keys 8nt + 2tig..
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack_h2(p2, p3);   // row g+8
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < KC / 16; ++kk) {
#pragma unroll
      for (int dt = 0; dt < NDT; dt += 2) {
        uint32_t r[4];
        ldsm_x4_t(r, &Vs[16 * kk + 8 * (mi & 1) + ri][8 * dt + 8 * (mi >> 1)]);
        mma16816(oacc[dt], pa[kk], r[0], r[1]);
        mma16816(oacc[dt + 1], pa[kk], r[2], r[3]);
      }
    }
  }

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = 1.0f / l0, inv1 = 1.0f / l1;
  const int64_t r0 = wr0 + g, r1 = wr0 + g + 8;
#pragma unroll
  for (int dt = 0; dt < NDT; ++dt) {
    const int c = h * D + 8 * dt + 2 * tig;
    if (r0 < a.s)
      *reinterpret_cast<__half2*>(a.out + (bi * a.s + r0) * a.ldo + c) =
          __floats2half2_rn(oacc[dt][0] * inv0, oacc[dt][1] * inv0);
    if (r1 < a.s)
      *reinterpret_cast<__half2*>(a.out + (bi * a.s + r1) * a.ldo + c) =
          __floats2half2_rn(oacc[dt][2] * inv1, oacc[dt][3] * inv1);
  }
}

template <int D>
fg_status launch_prefill_mma(const fg_kv& kv, const void* q, int64_t ldq, int64_t b, int64_t s, void* out,
                             int64_t ldo, cudaStream_t st) {
  PrefillArgs a;
  a.kc = reinterpret_cast<const uint32_t*>(kv.k_codes);
  a.vc = reinterpret_cast<const uint32_t*>(kv.v_codes);
  a.kmin = kv.k_mins;
  a.kscale = kv.k_scales;
  a.vmin = kv.v_mins;
  a.vscale = kv.v_scales;
  a.q = static_cast<const __half*>(q);
  a.ldq = ldq;
  a.out = static_cast<__half*>(out);
  a.ldo = ldo;
  a.s = s;
  a.heads = kv.heads;
  a.cap = kv.capacity;
  const int64_t nqb = (s + QB - 1) / QB;
  Trace tr(KC_ATTN_PREFILL, st);
  prefill_attn_mma_kernel<D><<<static_cast<unsigned>(b * kv.heads * nqb), 128, 0, st>>>(a);
  return check_launch("prefill_attn_mma_kernel");
}

}  // namespace

fg_status prefill_attention(const fg_kv& kv, const void* q, int64_t ldq, int64_t b, int64_t s, void* out,
                            int64_t ldo, cudaStream_t st) {
  if (b == 0 || s == 0) return FG_OK;
  if (kv.codec == FG_CODEC_Q4G64 && kv.dtype == FG_F16) {
    if (kv.head_dim == 128) return launch_prefill_mma<128>(kv, q, ldq, b, s, out, ldo, st);
    if (kv.head_dim == 64) return launch_prefill_mma<64>(kv, q, ldq, b, s, out, ldo, st);
  }
  return prefill_attention_simt(kv, q, ldq, b, s, out, ldo, st);
}

}  // namespace fg
