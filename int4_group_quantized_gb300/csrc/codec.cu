// The 4-bit group codec (FlexGen notes, "5. 近似方法", group-wise quantization
// equation, b = 4, g = 64) and the KV-cache writes that use it.
//
// Every operation of the quantizer is an explicitly rounded fp32 intrinsic
// (__fsub_rn, __fdiv_rn, __fmul_rn, rintf), so nothing can be contracted into
// an FMA and the codes are bit-identical to an IEEE fp32 evaluation of
// ((x - min) / (max - min)) * 15 rounded half-to-even.
//
// Layout of the work: a group of 64 consecutive elements is spread over 8
// consecutive lanes, 8 elements each (one 16-byte load of fp16, two of fp32);
// the group min/max is reduced with three xor-shuffles on order-preserving
// integer keys, which makes the result independent of reduction order and
// gives -0 < +0.  Each lane writes one 32-bit word of codes (8 nibbles); the
// first lane of the group writes (min, scale).
#include "codec_dev.cuh"
#include "fg_internal.cuh"

namespace fg {
namespace {

using codec::quantize_group8;

__device__ __forceinline__ void load8(const __half* p, float (&v)[8]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(p);
  const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void store8(__half* p, const float (&v)[8]) {
  uint4 raw;
  __half2* h = reinterpret_cast<__half2*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = raw;
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// x viewed as ngroups consecutive groups of 64.
template <typename T>
__global__ void __launch_bounds__(256) quantize_kernel(const T* __restrict__ x, int64_t ngroups,
                                                       uint32_t* __restrict__ codes,
                                                       float* __restrict__ mins,
                                                       float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int part = lane & 7;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t base = warp * 4; base < ngroups; base += nwarps * 4) {
    const int64_t g = base + (lane >> 3);
    const bool valid = g < ngroups;
    float v[8];
    if (valid) {
      load8(x + g * 64 + part * 8, v);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(0x7fffffffu);
    }
    float mn, sc;
    const uint32_t packed = quantize_group8(v, mn, sc);
    if (valid) {
      codes[g * 8 + part] = packed;
      if (part == 0) {
        mins[g] = mn;
        scales[g] = sc;
      }
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) dequant_kernel(const uint32_t* __restrict__ codes,
                                                      const float* __restrict__ mins,
                                                      const float* __restrict__ scales,
                                                      int64_t nwords, T* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; w < nwords;
       w += stride) {
    const uint32_t c = codes[w];
    const int64_t g = w >> 3;  // 8 words of codes per group
    const float mn = mins[g], sc = scales[g];
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __fmaf_rn(static_cast<float>((c >> (4 * i)) & 15u), sc, mn);
    store8(out + w * 8, v);
  }
}

// KV rows of T tokens per sequence -> cache slots pos0..pos0+T-1.  One
// quantization group = 64 hidden values of one token of one of K/V.
struct KVDst {
  uint32_t* codes[2];
  float* mins[2];
  float* scales[2];
};

// A warp owns one (K or V, sequence, head) and a run of kKvTokens
// consecutive tokens, so that the codes and (min, scale) pairs it writes are
// contiguous in the cache (slot-major per head): 8 lanes per 64-group, the
// groups of a head row side by side, 32 / (8 * groups per head) tokens at
// a time, kKvBatches such batches in flight (four measured slower: fewer
// warps fit).
constexpr int kKvTokens = 32;
constexpr int kKvBatches = 2;

template <typename T, int NG>
__global__ void __launch_bounds__(256) kv_store_q4_kernel(const T* __restrict__ ksrc,
                                                          const T* __restrict__ vsrc, int64_t ld,
                                                          int64_t b, int64_t ntok, int64_t pos0,
                                                          int heads, int64_t cap, KVDst dst, int write_back) {
  constexpr int D = 64 * NG;
  constexpr int kTpi = 4 / NG;   // tokens per warp-wide batch
  const int lane = threadIdx.x & 31;
  const int part = lane & 7, gi = (lane >> 3) % NG, tb = lane / (8 * NG);
  const int64_t chunks = (ntok + kKvTokens - 1) / kKvTokens;
  const int64_t items = 2 * b * heads * chunks;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t it = warp; it < items; it += nwarps) {
    const int64_t ch = it % chunks;
    const int64_t bh = (it / chunks) % (b * heads);
    const int which = static_cast<int>(it / (chunks * b * heads));
    const int64_t bi = bh / heads;
    const int h = static_cast<int>(bh % heads);
    const int64_t t0 = ch * kKvTokens, t1 = min(ntok, t0 + kKvTokens);
    const T* src = (which ? vsrc : ksrc) + (bi * ntok) * ld + h * D + gi * 64 + part * 8;
    const int64_t slot0 = bh * cap + pos0;
    uint32_t* codes = which ? dst.codes[1] : dst.codes[0];   // selects: no local copy of the parameter
    float* mins = which ? dst.mins[1] : dst.mins[0];
    float* scales = which ? dst.scales[1] : dst.scales[0];
    for (int64_t tt = t0; tt < t1; tt += kKvBatches * kTpi) {
      float v[kKvBatches][8];
#pragma unroll
      for (int u = 0; u < kKvBatches; ++u) {
        const int64_t ti = tt + u * kTpi + tb;
        if (ti < t1) {
          load8(src + ti * ld, v[u]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) v[u][e] = 0.0f;
        }
      }
#pragma unroll
      for (int u = 0; u < kKvBatches; ++u) {
        const int64_t ti = tt + u * kTpi + tb;
        float mn, sc;
        const uint32_t packed = quantize_group8(v[u], mn, sc);   // every lane of the group takes part
        if (ti < t1) {
          const int64_t slot = slot0 + ti;
          codes[(slot * (D / 2) + gi * 32) / 4 + part] = packed;
          if (part == 0) {
            mins[slot * NG + gi] = mn;
            scales[slot * NG + gi] = sc;
          }
          if (write_back) {
            // the values attention reads back from the cache, fp16(fmaf(q,
            // scale, min)), in place of the row just quantized
            float r[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) r[e] = __fmaf_rn(codec::code_float((packed >> (4 * e)) & 15u), sc, mn);
            store8(const_cast<T*>(src) + ti * ld, r);
          }
        }
      }
    }
  }
}

// Codec off: copy rows into the dense cache, 8 elements per thread.
template <typename T>
__global__ void kv_store_dense_kernel(const T* __restrict__ ksrc, const T* __restrict__ vsrc,
                                      int64_t ld, int64_t b, int64_t ntok, int64_t pos0, int h1,
                                      int heads, int d, int64_t cap, T* kd, T* vd) {
  const int64_t n8 = 2 * b * ntok * (h1 / 8);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += stride) {
    const int c8 = static_cast<int>(i % (h1 / 8));
    const int64_t rest = i / (h1 / 8);
    const int64_t row = rest % (b * ntok);
    const int which = static_cast<int>(rest / (b * ntok));
    const int64_t bi = row / ntok, ti = row % ntok;
    float v[8];
    load8((which ? vsrc : ksrc) + row * ld + c8 * 8, v);
    const int col = c8 * 8, head = col / d, dd = col % d;
    T* out = which ? vd : kd;
    store8(out + ((bi * heads + head) * cap + pos0 + ti) * d + dd, v);
  }
}

int grid_for(int64_t items, int per_block) {
  const int64_t want = (items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
  return static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
}

}  // namespace

fg_status quantize_rows(const void* x, fg_dtype dt, int64_t rows, int64_t cols, uint8_t* codes,
                        float* mins, float* scales, cudaStream_t st) {
  const int64_t ngroups = rows * (cols / 64);
  if (ngroups == 0) return FG_OK;
  const int grid = grid_for(ngroups, 32);  // 8 warps x 4 groups per block
  Trace tr(KC_QUANTIZE, st);
  if (dt == FG_F16)
    quantize_kernel<__half><<<grid, 256, 0, st>>>(static_cast<const __half*>(x), ngroups,
                                                  reinterpret_cast<uint32_t*>(codes), mins, scales);
  else
    quantize_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(x), ngroups,
                                                 reinterpret_cast<uint32_t*>(codes), mins, scales);
  return check_launch("quantize_kernel");
}

fg_status dequant_rows(const uint8_t* codes, const float* mins, const float* scales,
                       int64_t rows, int64_t cols, void* out, fg_dtype dt, cudaStream_t st) {
  const int64_t nwords = rows * cols / 8;
  if (nwords == 0) return FG_OK;
  const int grid = grid_for(nwords, 256);
  Trace tr(KC_DEQUANT, st);
  const uint32_t* c = reinterpret_cast<const uint32_t*>(codes);
  if (dt == FG_F16)
    dequant_kernel<__half><<<grid, 256, 0, st>>>(c, mins, scales, nwords, static_cast<__half*>(out));
  else
    dequant_kernel<float><<<grid, 256, 0, st>>>(c, mins, scales, nwords, static_cast<float*>(out));
  return check_launch("dequant_kernel");
}

fg_status kv_store(const fg_kv& kv, const void* ksrc, const void* vsrc, int64_t ld, int64_t b,
                   int64_t ntok, int64_t pos0, cudaStream_t st, bool write_back) {
  const int h1 = kv.heads * kv.head_dim;
  if (b == 0 || ntok == 0) return FG_OK;
  if (kv.codec == FG_CODEC_Q4G64) {
    if (kv.head_dim != 64 && kv.head_dim != 128)
      return fail(FG_ERR_UNSUPPORTED, "4-bit cache with head_dim %d (64 or 128)", kv.head_dim);
    KVDst dst;
    dst.codes[0] = reinterpret_cast<uint32_t*>(kv.k_codes);
    dst.codes[1] = reinterpret_cast<uint32_t*>(kv.v_codes);
    dst.mins[0] = kv.k_mins;
    dst.mins[1] = kv.v_mins;
    dst.scales[0] = kv.k_scales;
    dst.scales[1] = kv.v_scales;
    const int64_t items = 2 * b * kv.heads * ((ntok + kKvTokens - 1) / kKvTokens);
    const int grid = grid_for(items, 8);   // a (K/V, sequence, head, token run) per warp, 8 warps per block
    Trace tr(KC_KV_STORE, st);
    const bool wide = kv.head_dim == 128;
    if (kv.dtype == FG_F16) {
      const __half* k = static_cast<const __half*>(ksrc);
      const __half* v = static_cast<const __half*>(vsrc);
      if (wide)
        kv_store_q4_kernel<__half, 2><<<grid, 256, 0, st>>>(k, v, ld, b, ntok, pos0, kv.heads, kv.capacity, dst, write_back ? 1 : 0);
      else
        kv_store_q4_kernel<__half, 1><<<grid, 256, 0, st>>>(k, v, ld, b, ntok, pos0, kv.heads, kv.capacity, dst, write_back ? 1 : 0);
    } else {
      const float* k = static_cast<const float*>(ksrc);
      const float* v = static_cast<const float*>(vsrc);
      if (wide)
        kv_store_q4_kernel<float, 2><<<grid, 256, 0, st>>>(k, v, ld, b, ntok, pos0, kv.heads, kv.capacity, dst, write_back ? 1 : 0);
      else
        kv_store_q4_kernel<float, 1><<<grid, 256, 0, st>>>(k, v, ld, b, ntok, pos0, kv.heads, kv.capacity, dst, write_back ? 1 : 0);
    }
    return check_launch("kv_store_q4_kernel");
  }
  const int64_t n8 = 2 * b * ntok * (h1 / 8);
  const int grid = grid_for(n8, 256);
  Trace tr(KC_KV_STORE, st);
  if (kv.dtype == FG_F16)
    kv_store_dense_kernel<__half><<<grid, 256, 0, st>>>(
        static_cast<const __half*>(ksrc), static_cast<const __half*>(vsrc), ld, b, ntok, pos0, h1,
        kv.heads, kv.head_dim, kv.capacity, static_cast<__half*>(kv.k_dense),
        static_cast<__half*>(kv.v_dense));
  else
    kv_store_dense_kernel<float><<<grid, 256, 0, st>>>(
        static_cast<const float*>(ksrc), static_cast<const float*>(vsrc), ld, b, ntok, pos0, h1,
        kv.heads, kv.head_dim, kv.capacity, static_cast<float*>(kv.k_dense),
        static_cast<float*>(kv.v_dense));
  return check_launch("kv_store_dense_kernel");
}

}  // namespace fg

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
using fg::aligned;
using fg::fail;

extern "C" fg_status fg_quantize_g64(const void* x, fg_dtype dt, int64_t rows, int64_t cols,
                                     uint8_t* codes, float* mins, float* scales,
                                     cudaStream_t stream) {
  if (dt != FG_F16 && dt != FG_F32) return fail(FG_ERR_ARG, "dtype %d", static_cast<int>(dt));
  if (rows < 0 || cols < 0) return fail(FG_ERR_ARG, "negative size");
  if (cols % 64 != 0) return fail(FG_ERR_SHAPE, "cols %lld is not a multiple of 64", (long long)cols);
  if (rows == 0 || cols == 0) return FG_OK;
  if (!x || !codes || !mins || !scales) return fail(FG_ERR_ARG, "null pointer");
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(mins, 4) || !aligned(scales, 4))
    return fail(FG_ERR_ALIGN, "x and codes need 16-byte, mins/scales 4-byte alignment");
  return fg::quantize_rows(x, dt, rows, cols, codes, mins, scales, stream);
}

extern "C" fg_status fg_dequant_g64(const uint8_t* codes, const float* mins, const float* scales,
                                    int64_t rows, int64_t cols, void* out, fg_dtype dt,
                                    cudaStream_t stream) {
  if (dt != FG_F16 && dt != FG_F32) return fail(FG_ERR_ARG, "dtype %d", static_cast<int>(dt));
  if (rows < 0 || cols < 0) return fail(FG_ERR_ARG, "negative size");
  if (cols % 64 != 0) return fail(FG_ERR_SHAPE, "cols %lld is not a multiple of 64", (long long)cols);
  if (rows == 0 || cols == 0) return FG_OK;
  if (!out || !codes || !mins || !scales) return fail(FG_ERR_ARG, "null pointer");
  if (!aligned(out, 16) || !aligned(codes, 16) || !aligned(mins, 4) || !aligned(scales, 4))
    return fail(FG_ERR_ALIGN, "out and codes need 16-byte, mins/scales 4-byte alignment");
  return fg::dequant_rows(codes, mins, scales, rows, cols, out, dt, stream);
}
