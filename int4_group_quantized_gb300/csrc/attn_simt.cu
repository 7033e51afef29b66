// CUDA-core attention over the KV cache (FlexGen notes, "背景知识": decode
// t_Out = Softmax(t_Q x_K^T / sqrt(h1)) x_V, prefill with the same form over
// the prompt; "5. 近似方法": K/V stored in 4-bit groups and converted back to
// the compute type before use).
//
// These kernels read K/V through the codec exactly like the tensor-core
// kernels and serve the fp32 activation type and caches without the codec.
// Softmax is evaluated online (running max and sum, chunk by chunk), which is
// the same function as the max-subtracted softmax of the oracle.
#include <math.h>

#include "fg_internal.cuh"

namespace fg {
namespace {

constexpr unsigned kFull = 0xffffffffu;

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <typename T> __device__ __forceinline__ float round_to(float v) { return to_f<T>(from_f<T>(v)); }

struct KVSrc {
  const uint32_t* codes[2];  // K, V; 8 codes per word
  const float* mins[2];
  const float* scales[2];
  const void* dense[2];
};

// 8 consecutive values (dims 8w..8w+7) of row `slot` of K (which=0) or V.
template <typename T, bool QUANT, int D>
__device__ __forceinline__ void load_kv8(const KVSrc& kv, int which, int64_t slot, int w,
                                         float (&v)[8]) {
  if (QUANT) {
    const uint32_t c = kv.codes[which][slot * (D / 8) + w];
    const int64_t g = slot * (D / 64) + (w >> 3);
    const float mn = kv.mins[which][g], sc = kv.scales[which][g];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      v[i] = round_to<T>(__fmaf_rn(static_cast<float>((c >> (4 * i)) & 15u), sc, mn));
  } else {
    const T* p = static_cast<const T*>(kv.dense[which]) + slot * D + w * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = to_f<T>(p[i]);
  }
}

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float o = __shfl_xor_sync(kFull, v, off);
    v = is_max ? fmaxf(v, o) : v + o;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  float r = red[0];
  for (int i = 1; i < nw; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
  return r;
}

// One CTA per (sequence, head); 128 threads = (128 / (D/8)) token lanes of
// D/8 threads, each thread owning 8 dims of a token row.
template <typename T, bool QUANT, int D>
__global__ void __launch_bounds__(128) decode_attn_simt_kernel(KVSrc kv, const T* __restrict__ q,
                                                               int64_t ldq, int64_t pos,
                                                               T* __restrict__ out, int64_t ldo,
                                                               int heads, int64_t cap) {
  constexpr int TPR = D / 8;
  constexpr int NTL = 128 / TPR;
  constexpr int CH = 256;
  __shared__ float qs[D];
  __shared__ float ps[CH];
  __shared__ float red[4];
  __shared__ float accs[NTL][D];
  const int bh = blockIdx.x;
  const int64_t bi = bh / heads;
  const int h = bh % heads;
  const int tid = threadIdx.x, tl = tid / TPR, dl = tid % TPR;
  const float qscale = 1.0f / sqrtf(static_cast<float>(D));
  for (int i = tid; i < D; i += 128) qs[i] = to_f<T>(q[bi * ldq + h * D + i]) * qscale;
  __syncthreads();
  float qr[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) qr[i] = qs[dl * 8 + i];
  const int64_t slot0 = (bi * heads + h) * cap;
  const int64_t len = pos + 1;
  float run_max = -INFINITY, run_sum = 0.0f, acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;

  for (int64_t c0 = 0; c0 < len; c0 += CH) {
    const int n = static_cast<int>(len - c0 < CH ? len - c0 : CH);
    for (int jb = 0; jb < n; jb += NTL) {
      const int j = jb + tl;
      float part = 0.0f;
      if (j < n) {
        float kr[8];
        load_kv8<T, QUANT, D>(kv, 0, slot0 + c0 + j, dl, kr);
#pragma unroll
        for (int i = 0; i < 8; ++i) part = fmaf(qr[i], kr[i], part);
      }
#pragma unroll
      for (int off = TPR / 2; off > 0; off >>= 1) part += __shfl_xor_sync(kFull, part, off);
      if (j < n && dl == 0) ps[j] = part;
    }
    __syncthreads();
    float m = -INFINITY;
    for (int j = tid; j < n; j += 128) m = fmaxf(m, ps[j]);
    const float cmax = block_reduce(m, true, red);
    const float new_max = fmaxf(run_max, cmax);
    const float alpha = expf(run_max - new_max);
    float sl = 0.0f;
    for (int j = tid; j < n; j += 128) {
      const float p = expf(ps[j] - new_max);
      ps[j] = p;
      sl += p;
    }
    const float csum = block_reduce(sl, false, red);  // its barriers also publish ps
    run_sum = run_sum * alpha + csum;
    run_max = new_max;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] *= alpha;
    for (int j = tl; j < n; j += NTL) {
      float vr[8];
      load_kv8<T, QUANT, D>(kv, 1, slot0 + c0 + j, dl, vr);
      const float p = ps[j];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(p, vr[i], acc[i]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) accs[tl][dl * 8 + i] = acc[i];
  __syncthreads();
  for (int i = tid; i < D; i += 128) {
    float s = 0.0f;
#pragma unroll
    for (int t = 0; t < NTL; ++t) s += accs[t][i];
    out[bi * ldo + h * D + i] = from_f<T>(s / run_sum);
  }
}

// Causal prefill: one CTA per (sequence, head, 16 queries); 8 threads per
// query.  Keys are staged 32 at a time in shared memory, dequantized.
template <typename T, bool QUANT, int D>
__global__ void __launch_bounds__(128) prefill_attn_simt_kernel(KVSrc kv, const T* __restrict__ q,
                                                                int64_t ldq, int64_t s,
                                                                T* __restrict__ out, int64_t ldo,
                                                                int heads, int64_t cap) {
  constexpr int QB = 16, KC = 32, SUB = 8;
  constexpr int DPT = D / SUB;  // output dims per thread
  __shared__ float Qs[QB][D + 4];
  __shared__ float Ks[KC][D + 1];
  __shared__ float Vs[KC][D + 1];
  __shared__ float Ps[QB][KC + 1];
  const int64_t nqb = (s + QB - 1) / QB;
  const int64_t qb = blockIdx.x % nqb;
  const int64_t bh = blockIdx.x / nqb;
  const int64_t bi = bh / heads;
  const int h = static_cast<int>(bh % heads);
  const int tid = threadIdx.x, qi = tid / SUB, sub = tid % SUB;
  const int64_t q0 = qb * QB;
  const float qscale = 1.0f / sqrtf(static_cast<float>(D));
  for (int i = tid; i < QB * D; i += 128) {
    const int r = i / D, c = i % D;
    const int64_t qa = q0 + r;
    Qs[r][c] = qa < s ? to_f<T>(q[(bi * s + qa) * ldq + h * D + c]) * qscale : 0.0f;
  }
  const int64_t my_q = q0 + qi;
  const int64_t kend = (q0 + QB < s ? q0 + QB : s);  // keys 0..kend-1 are visible to someone
  const int64_t slot0 = (bi * heads + h) * cap;
  float run_max = -INFINITY, run_sum = 0.0f, acc[DPT];
#pragma unroll
  for (int i = 0; i < DPT; ++i) acc[i] = 0.0f;

  for (int64_t c0 = 0; c0 < kend; c0 += KC) {
    __syncthreads();
    for (int i = tid; i < KC * (D / 8); i += 128) {
      const int r = i / (D / 8), w = i % (D / 8);
      float kr[8], vr[8];
      if (c0 + r < kend) {
        load_kv8<T, QUANT, D>(kv, 0, slot0 + c0 + r, w, kr);
        load_kv8<T, QUANT, D>(kv, 1, slot0 + c0 + r, w, vr);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) kr[e] = vr[e] = 0.0f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        Ks[r][w * 8 + e] = kr[e];
        Vs[r][w * 8 + e] = vr[e];
      }
    }
    __syncthreads();
    float sc[KC / SUB];
    float m = -INFINITY;
#pragma unroll
    for (int t = 0; t < KC / SUB; ++t) {
      const int j = sub + SUB * t;
      float d = 0.0f;
#pragma unroll 16
      for (int e = 0; e < D; ++e) d = fmaf(Qs[qi][e], Ks[j][e], d);
      const bool vis = (c0 + j <= my_q) && (c0 + j < kend);
      sc[t] = vis ? d : -INFINITY;
      m = fmaxf(m, sc[t]);
    }
#pragma unroll
    for (int off = SUB / 2; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
    const float new_max = fmaxf(run_max, m);
    // a query below this whole chunk keeps its state (new_max stays finite
    // from chunk 0, which always holds key 0)
    const float alpha = expf(run_max - new_max);
    float sl = 0.0f;
#pragma unroll
    for (int t = 0; t < KC / SUB; ++t) {
      const float p = expf(sc[t] - new_max);
      Ps[qi][sub + SUB * t] = p;
      sl += p;
    }
#pragma unroll
    for (int off = SUB / 2; off > 0; off >>= 1) sl += __shfl_xor_sync(kFull, sl, off);
    run_sum = run_sum * alpha + sl;
    run_max = new_max;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < DPT; ++i) acc[i] *= alpha;
    for (int j = 0; j < KC; ++j) {
      const float p = Ps[qi][j];
#pragma unroll
      for (int i = 0; i < DPT; ++i) acc[i] = fmaf(p, Vs[j][sub + SUB * i], acc[i]);
    }
  }
  if (my_q < s) {
    const float inv = 1.0f / run_sum;
#pragma unroll
    for (int i = 0; i < DPT; ++i)
      out[(bi * s + my_q) * ldo + h * D + sub + SUB * i] = from_f<T>(acc[i] * inv);
  }
}

KVSrc make_src(const fg_kv& kv) {
  KVSrc s;
  s.codes[0] = reinterpret_cast<const uint32_t*>(kv.k_codes);
  s.codes[1] = reinterpret_cast<const uint32_t*>(kv.v_codes);
  s.mins[0] = kv.k_mins;
  s.mins[1] = kv.v_mins;
  s.scales[0] = kv.k_scales;
  s.scales[1] = kv.v_scales;
  s.dense[0] = kv.k_dense;
  s.dense[1] = kv.v_dense;
  return s;
}

template <typename T, bool QUANT, int D>
void launch_decode(const fg_kv& kv, const void* q, int64_t ldq, int64_t b, int64_t pos, void* out,
                   int64_t ldo, cudaStream_t st) {
  Trace tr(KC_ATTN_DECODE, st);
  decode_attn_simt_kernel<T, QUANT, D><<<static_cast<unsigned>(b * kv.heads), 128, 0, st>>>(
      make_src(kv), static_cast<const T*>(q), ldq, pos, static_cast<T*>(out), ldo, kv.heads,
      kv.capacity);
}

template <typename T, bool QUANT, int D>
void launch_prefill(const fg_kv& kv, const void* q, int64_t ldq, int64_t b, int64_t s, void* out,
                    int64_t ldo, cudaStream_t st) {
  const int64_t nqb = (s + 15) / 16;
  Trace tr(KC_ATTN_PREFILL, st);
  prefill_attn_simt_kernel<T, QUANT, D><<<static_cast<unsigned>(b * kv.heads * nqb), 128, 0, st>>>(
      make_src(kv), static_cast<const T*>(q), ldq, s, static_cast<T*>(out), ldo, kv.heads,
      kv.capacity);
}

}  // namespace

fg_status decode_attention_simt(const fg_kv& kv, const void* q, int64_t ldq, int64_t b,
                                int64_t pos, void* out, int64_t ldo, cudaStream_t st) {
  if (b == 0) return FG_OK;
  const bool qz = kv.codec == FG_CODEC_Q4G64;
  const bool h = kv.dtype == FG_F16;
  if (kv.head_dim == 64) {
    if (h) (qz ? launch_decode<__half, true, 64> : launch_decode<__half, false, 64>)(kv, q, ldq, b, pos, out, ldo, st);
    else (qz ? launch_decode<float, true, 64> : launch_decode<float, false, 64>)(kv, q, ldq, b, pos, out, ldo, st);
  } else {
    if (h) (qz ? launch_decode<__half, true, 128> : launch_decode<__half, false, 128>)(kv, q, ldq, b, pos, out, ldo, st);
    else (qz ? launch_decode<float, true, 128> : launch_decode<float, false, 128>)(kv, q, ldq, b, pos, out, ldo, st);
  }
  return check_launch("decode_attn_simt_kernel");
}

fg_status prefill_attention_simt(const fg_kv& kv, const void* q, int64_t ldq, int64_t b, int64_t s,
                                 void* out, int64_t ldo, cudaStream_t st) {
  if (b == 0 || s == 0) return FG_OK;
  const bool qz = kv.codec == FG_CODEC_Q4G64;
  const bool h = kv.dtype == FG_F16;
  if (kv.head_dim == 64) {
    if (h) (qz ? launch_prefill<__half, true, 64> : launch_prefill<__half, false, 64>)(kv, q, ldq, b, s, out, ldo, st);
    else (qz ? launch_prefill<float, true, 64> : launch_prefill<float, false, 64>)(kv, q, ldq, b, s, out, ldo, st);
  } else {
    if (h) (qz ? launch_prefill<__half, true, 128> : launch_prefill<__half, false, 128>)(kv, q, ldq, b, s, out, ldo, st);
    else (qz ? launch_prefill<float, true, 128> : launch_prefill<float, false, 128>)(kv, q, ldq, b, s, out, ldo, st);
  }
  return check_launch("prefill_attn_simt_kernel");
}

}  // namespace fg
