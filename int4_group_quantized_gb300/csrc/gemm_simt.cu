// CUDA-core products Y = epilogue(X . W) with the 4-bit weights dequantized
// on the fly (FlexGen notes, "5. 近似方法": weights stored quantized and
// converted back to FP16 before compute; "背景知识": the layer's x . w
// products, ReLU and residual adds).
//
// This path serves every product the tensor-core kernels do not take: the
// fp32 activation type, and blocks too small to fill a tensor-core tile.
// Tile 64 x 64 x 32 per 256-thread CTA, 4 x 4 outputs per thread, fp32
// accumulation.  A 64-column tile is exactly one quantization group of a
// weight row, so each weight row of the tile needs one (min, scale) pair.
#include "fg_internal.cuh"

namespace fg {
namespace {

__device__ __forceinline__ void ld8(const __half* p, float (&v)[8]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(p);
  const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void ld8(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
// Rounds a dequantized weight to the compute type (fp16 layers compute on
// fp16 weights).
template <typename T> __device__ __forceinline__ float round_to(float v) { return to_f<T>(from_f<T>(v)); }

constexpr int BM = 64, BN = 64, BK = 32;

template <typename T, bool QUANT>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs a) {
  __shared__ __align__(16) float Xs[BK][BM + 4];
  __shared__ __align__(16) float Ws[BK][BN + 4];
  const int tid = threadIdx.x;
  const int64_t ncol = static_cast<int64_t>(blockIdx.x) * BN;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BM;
  int s = 0;
  while (s + 1 < a.nseg && ncol >= a.seg[s + 1].n0) ++s;
  const WSeg& seg = a.seg[s];
  const int64_t nl = ncol - seg.n0;
  const T* X = static_cast<const T*>(a.X);
  const int tx = tid & 15, ty = tid >> 4;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  for (int64_t k0 = 0; k0 < a.K; k0 += BK) {
    {
      const int r = tid >> 2, kk = (tid & 3) * 8;
      const int64_t m = m0 + r;
      float v[8];
      if (m < a.M) {
        ld8(X + m * a.ldx + k0 + kk, v);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) Xs[kk + i][r] = v[i];
    }
    {
      const int kr = tid >> 3, nn = (tid & 7) * 8;
      const int64_t k = k0 + kr;
      float w[8];
      if (QUANT) {
        const uint32_t c = *reinterpret_cast<const uint32_t*>(seg.codes + k * (seg.N / 2) + (nl + nn) / 2);
        const int64_t gi = k * (seg.N / 64) + nl / 64;
        const float mn = seg.mins[gi], sc = seg.scales[gi];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w[i] = round_to<T>(__fmaf_rn(static_cast<float>((c >> (4 * i)) & 15u), sc, mn));
      } else {
        ld8(static_cast<const T*>(seg.dense) + k * seg.N + nl + nn, w);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) Ws[kr][nn + i] = w[i];
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      const float4 xa = *reinterpret_cast<const float4*>(&Xs[kk][ty * 4]);
      const float4 wb = *reinterpret_cast<const float4*>(&Ws[kk][tx * 4]);
      const float xv[4] = {xa.x, xa.y, xa.z, xa.w};
      const float wv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }

  T* Y = static_cast<T*>(a.Y);
  const T* R = static_cast<const T*>(a.R);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = ncol + tx * 4 + j;
      float v = acc[i][j];
      if (R) v += to_f<T>(R[m * a.ldr + n]);
      if (a.relu) v = fmaxf(v, 0.0f);
      Y[m * a.ldy + n] = from_f<T>(v);
    }
  }
}

}  // namespace

fg_status gemm_simt(const GemmArgs& a, cudaStream_t st) {
  if (a.M == 0 || a.N == 0) return FG_OK;
  dim3 grid(static_cast<unsigned>(a.N / BN), static_cast<unsigned>((a.M + BM - 1) / BM));
  Trace tr(KC_GEMM_SIMT, st);
  if (a.dtype == FG_F16) {
    if (a.quant) gemm_simt_kernel<__half, true><<<grid, 256, 0, st>>>(a);
    else gemm_simt_kernel<__half, false><<<grid, 256, 0, st>>>(a);
  } else {
    if (a.quant) gemm_simt_kernel<float, true><<<grid, 256, 0, st>>>(a);
    else gemm_simt_kernel<float, false><<<grid, 256, 0, st>>>(a);
  }
  return check_launch("gemm_simt_kernel");
}

}  // namespace fg
