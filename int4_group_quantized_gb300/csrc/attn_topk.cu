// Top-K sparse decode attention over the 4-bit KV cache (FlexGen notes,
// "5. 近似方法", sparse attention: once the attention matrix is computed,
// each query keeps the indices of its Top-K tokens in the K cache, the other
// tokens are dropped, and only those rows of the V cache are read).
//
// One CTA (4 warps) per (sequence, head), all tokens 0..pos visible:
//   1. scores.  Every K row is read, 16-token blocks per warp.  Unlike the
//      dense kernel, each K value is first restored exactly as the format
//      gives it, fp16(fmaf(c, scale, min)) ("converted back to FP16 before
//      compute"), so that the scores, which decide which tokens are kept,
//      differ from exact arithmetic on those fp16 values only by the fp32
//      accumulation of the warp-level MMA (exact fp16 products).  The
//      base-2 scores of all tokens stay in shared memory.
//   2. softmax over all tokens: the maximum, then the sum of exp2(s - max),
//      each reduced in a fixed order.
//   3. selection.  An MSB-first radix select over the scores' order-
//      preserving 32-bit keys (four 8-bit digits, a shared histogram per
//      digit) finds the keep-th largest key T and how many keys equal to T
//      are taken; those are the lowest-indexed ones (ties rank by index).
//      The selected tokens are listed in index order with two CTA scans.
//   4. values.  Only the listed V rows are read: each weight
//      p_i = exp2(s_i - max) / sum is applied to the value the format
//      restores, fp16(fmaf(c, scale, min)), accumulated in fp32 per warp in
//      list order and summed over the warps in warp order (deterministic).
// The kept weights are those of the softmax over all tokens; nothing is
// renormalised.
//
// Bytes per (sequence, head): every K row (d/2 code bytes + 8 bytes of
// (min, scale) per 64-group), keep V rows, q and the output.
#include <math.h>

#include "attn_dev.cuh"
#include "fg_internal.cuh"
#include "q4_dev.cuh"
#include "tc_ptx.cuh"

namespace fg {
namespace {

using namespace attn;
using namespace tc;

constexpr int kTopkWarps = 4;
constexpr int kTopkThreads = 32 * kTopkWarps;
constexpr int64_t kTopkMaxLen = 16384;   // scores + list in shared memory: 8 bytes per token
constexpr int kChunk = 128;              // tokens of K staged in shared memory at a time

// q of one (sequence, head) as this lane's m16n8k16 B fragments, in the
// order in which the K code words give their nibbles (the dense kernel's
// permutation, without its 1/16 on the upper nibbles): per group, the
// lane's dims 16*tig + 8w + (0,4 | 1,5) and (2,6 | 3,7).
template <int D>
__device__ __forceinline__ void setup_q_plain(uint32_t (&qb)[D / 64][4][2], const __half* qrow, int tig) {
#pragma unroll
  for (int g = 0; g < D / 64; ++g) {
    const uint4* src = reinterpret_cast<const uint4*>(qrow + g * 64 + 16 * tig);
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const uint4 raw = src[w];   // dims 16*tig + 8w .. +7, two per word
      const uint32_t lo01 = raw.x, lo23 = raw.y, lo45 = raw.z, lo67 = raw.w;
      qb[g][2 * w][0] = __byte_perm(lo01, lo45, 0x5410);       // (d0, d4)
      qb[g][2 * w][1] = __byte_perm(lo01, lo45, 0x7632);       // (d1, d5)
      qb[g][2 * w + 1][0] = __byte_perm(lo23, lo67, 0x5410);   // (d2, d6)
      qb[g][2 * w + 1][1] = __byte_perm(lo23, lo67, 0x7632);   // (d3, d7)
    }
  }
}

// One fp16x2 A register: the two codes that the lop3 placed as fp16
// (1024 + c) (hi = false) or (1024 + 16c) (hi = true), restored as
// fp16(fmaf(c, scale, min)) with the row's (scale, min).
template <bool HI>
__device__ __forceinline__ uint32_t restore_pair(uint32_t h, float2 s2, float2 m2) {
  const float2 c = HI ? q4::nib16_pair_f32(h) : q4::nib_pair_f32(h);
  return q4::cvt_f16x2(q4::fma_f32x2(c, s2, m2));
}

// Scores of tokens gq and gq+8 of a 16-token block, before the softmax
// scale, from the restored fp16 K values: sum over the groups of the MMA's
// dot products with q (qb from setup_q_plain).
template <int NG>
__device__ __forceinline__ void block_scores_f16(const uint32_t (&qb)[NG][4][2], const uint2 (&kw)[2][NG],
                                                 const float (&ksc)[2][NG], const float (&kmn)[2][NG], float& sc0,
                                                 float& sc1) {
  float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const float2 s0 = make_float2(ksc[0][g], ksc[0][g]), m0 = make_float2(kmn[0][g], kmn[0][g]);
    const float2 s1 = make_float2(ksc[1][g], ksc[1][g]), m1 = make_float2(kmn[1][g], kmn[1][g]);
#pragma unroll
    for (int w = 0; w < 2; ++w) {
#pragma unroll
      for (int sh = 0; sh < 2; ++sh) {   // bytes 0, 2 then bytes 1, 3 of the word
        const uint32_t x0 = (w ? kw[0][g].y : kw[0][g].x) >> (8 * sh);
        const uint32_t x1 = (w ? kw[1][g].y : kw[1][g].x) >> (8 * sh);
        mma16816(d, restore_pair<false>(lop_mask_or(x0, kLoNib, kMagic), s0, m0),
                 restore_pair<false>(lop_mask_or(x1, kLoNib, kMagic), s1, m1),
                 restore_pair<true>(lop_mask_or(x0, kHiNib, kMagic), s0, m0),
                 restore_pair<true>(lop_mask_or(x1, kHiNib, kMagic), s1, m1), qb[g][2 * w + sh][0],
                 qb[g][2 * w + sh][1]);
      }
    }
  }
  sc0 = d[0];
  sc1 = d[2];
}

// Order-preserving key: a > b as floats (no NaN) iff key(a) > key(b) as
// unsigned integers; -0 sorts just below +0.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum of v over the CTA's threads in thread order; the
// total goes to `total`.  Holds two CTA barriers (every thread calls it).
__device__ __forceinline__ int block_excl_scan(int v, int* wsum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kTopkWarps; ++w) {
    const int s = wsum[w];
    if (w < warp) base += s;
    tot += s;
  }
  __syncthreads();   // wsum is free for the next scan
  total = tot;
  return base + x - v;
}

// Shared memory of one CTA (dynamic): two staging buffers of kChunk tokens'
// K codes and their (scale, min) pairs, then the scores of all tokens and
// the list of kept tokens.
template <int D>
struct TopkLayout {
  static constexpr int NG = D / 64;
  static constexpr int kCodes = kChunk * D / 2;          // bytes of one chunk's codes
  static constexpr int kMeta = kChunk * NG * 2 * 4;      // its (scale, min) pairs
  static constexpr int kBuf = kCodes + kMeta;
  static constexpr int kFixed = 2 * kBuf + 16 * 2;       // + the two mbarriers
  static size_t bytes(int64_t len, int64_t nsel) { return kFixed + static_cast<size_t>(len + nsel) * 4; }
};

template <int D>
__global__ void __launch_bounds__(kTopkThreads, 8) decode_attn_topk_kernel(const DecodeArgs a, int keep,
                                                                         int32_t* __restrict__ idx_out) {
  constexpr int NG = D / 64;
  using Lay = TopkLayout<D>;
  extern __shared__ __align__(128) uint8_t dsm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(dsm + 2 * Lay::kBuf);   // chunk buffer b has landed
  float* sc = reinterpret_cast<float*>(dsm + Lay::kFixed);              // [len] base-2 scores
  __shared__ int hist[256];
  __shared__ int wsum[kTopkWarps];
  __shared__ float redf[kTopkWarps];
  __shared__ uint32_t sel_key;
  __shared__ int sel_need;
  __shared__ int abort_flag;
  __shared__ float red_o[kTopkWarps][D];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gq = lane >> 2, tig = lane & 3;
  const int bh = blockIdx.x;
  const int64_t bi = bh / a.heads;
  const int h = bh % a.heads;
  const int len = static_cast<int>(a.pos + 1);
  const int nsel = min(keep, len);
  const int64_t slot0 = static_cast<int64_t>(bh) * a.cap;
  int* list = reinterpret_cast<int*>(sc + len);
  volatile int* abort = &abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();

  tc::griddep_launch();
  tc::griddep_wait();

  if (a.knew != nullptr) {   // Concat first: the new token is one of the candidates
    if (warp == 0) {
      append_token<D>(a, slot0, bi, h, lane);
      tc::fence_proxy_async_global();   // the new row, then the bulk copies that read it
    }
    __syncthreads();
  }

  // ---- 1. scores of every token, K staged chunk by chunk ---------------------------
  uint32_t qb[NG][4][2];
  setup_q_plain<D>(qb, a.q + bi * a.ldq + h * D, tig);
  const int nch = (len + kChunk - 1) / kChunk;
  // chunk c into buffer c & 1: its codes by one bulk copy (thread 0), its
  // (scale, min) pairs by 4-byte asynchronous copies (all threads, one group)
  // Thread 0's record of the bulk copies: the last chunk it issued and the
  // last it saw land; after a wait gives up, no chunk is issued and the ones
  // in between are drained before the CTA leaves.
  int issued = -1, landed = -1;
  auto issue = [&](int c) {
    const int t0 = c * kChunk, n = min(kChunk, len - t0);
    uint8_t* buf = dsm + (c & 1) * Lay::kBuf;
    const bool go = !*abort;
    if (threadIdx.x == 0 && go) {
      mbar_expect_tx(&full[c & 1], static_cast<uint32_t>(n * (D / 2)));
      bulk_load(buf, a.kc + (slot0 + t0) * (D / 2), static_cast<uint32_t>(n * (D / 2)), &full[c & 1]);
      issued = c;
    }
    float* meta = reinterpret_cast<float*>(buf + Lay::kCodes);   // [tok][g][scale, min]
    if (go) {
      for (int e = threadIdx.x; e < n * NG; e += kTopkThreads) {
        const int64_t src = (slot0 + t0) * NG + e;
        cp_async4(meta + 2 * e, a.kscale + src);
        cp_async4(meta + 2 * e + 1, a.kmin + src);
      }
    }
    cp_async_commit();   // one group per chunk in every thread, empty or not
  };
  issue(0);
  {
    constexpr float kQs = score_scale_log2<D>();
    for (int c = 0; c < nch; ++c) {
      // buffer (c+1) & 1 was last read in chunk c-1, which ended with a CTA barrier
      if (c + 1 < nch) {
        issue(c + 1);
        cp_async_wait<1>();   // this thread's copies of chunk c are done
      } else {
        cp_async_wait<0>();
      }
      // one thread waits for the codes (the others would spend issue slots
      // polling); the CTA barrier then releases the rest
      if (threadIdx.x == 0 && !*abort && mbar_wait(&full[c & 1], (c >> 1) & 1, a.wait_limit, abort)) landed = c;
      __syncthreads();   // chunk c's codes have landed; every thread's pair copies are visible
      const int t0 = c * kChunk, n = min(kChunk, len - t0);
      const uint8_t* codes = dsm + (c & 1) * Lay::kBuf;
      const float* meta = reinterpret_cast<const float*>(codes + Lay::kCodes);
      if (!*abort) {
        for (int blk = warp; blk * 16 < n; blk += kTopkWarps) {
          uint2 kw[2][NG];
          float ksc[2][NG], kmn[2][NG];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int row = blk * 16 + gq + 8 * r;
#pragma unroll
            for (int g = 0; g < NG; ++g) {
              const bool v = row < n;
              kw[r][g] = v ? *reinterpret_cast<const uint2*>(codes + row * (D / 2) + g * 32 + 8 * tig)
                           : make_uint2(0u, 0u);
              ksc[r][g] = v ? meta[(row * NG + g) * 2] : 0.0f;
              kmn[r][g] = v ? meta[(row * NG + g) * 2 + 1] : 0.0f;
            }
          }
          float s0, s1;
          block_scores_f16<NG>(qb, kw, ksc, kmn, s0, s1);
          const int row = blk * 16 + gq;
          if (tig == 0) {
            if (row < n) sc[t0 + row] = s0 * kQs;
            if (row + 8 < n) sc[t0 + row + 8] = s1 * kQs;
          }
        }
      }
      __syncthreads();   // buffer c & 1 is free; the scores are visible
    }
  }
  if (*abort) {
    // a wait gave up: let every copy this CTA issued land before it leaves
    // (the output of this call is not meaningful; the host reads the error)
    if (threadIdx.x == 0) {
      volatile int dummy = 0;
      for (int c = landed + 1; c <= issued; ++c) mbar_wait(&full[c & 1], (c >> 1) & 1, kDrainLimit, &dummy);
      atomicOr(a.err, DEV_ERR_WAIT_TIMEOUT);
    }
    cp_async_wait<0>();
    return;
  }

  // ---- 2. softmax over all tokens: max, then sum of exp2(s - max) -----------------
  float M, L;
  {
    float m = -INFINITY;
    for (int i = threadIdx.x; i < len; i += kTopkThreads) m = fmaxf(m, sc[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) redf[warp] = m;
    __syncthreads();
    M = redf[0];
#pragma unroll
    for (int w = 1; w < kTopkWarps; ++w) M = fmaxf(M, redf[w]);
    __syncthreads();
    float l = 0.0f;
    for (int i = threadIdx.x; i < len; i += kTopkThreads) l += exp2f(sc[i] - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) redf[warp] = l;
    __syncthreads();
    L = 0.0f;
#pragma unroll
    for (int w = 0; w < kTopkWarps; ++w) L += redf[w];
  }

  // ---- 3. the nsel largest scores, ties to the lower index, listed in index order ----
  if (nsel < len) {
    uint32_t prefix = 0;
    int need = nsel;
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += kTopkThreads) hist[i] = 0;
      __syncthreads();
      for (int i = threadIdx.x; i < len; i += kTopkThreads) {
        const uint32_t k = order_key(sc[i]);
        if (shift == 24 || ((k ^ prefix) >> (shift + 8)) == 0) atomicAdd(&hist[(k >> shift) & 255u], 1);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l holds bins 255 - 8l down to 248 - 8l: a scan from the top
        int c[8], tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = hist[255 - 8 * lane - j];
          tot += c[j];
        }
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int before = incl - tot;
        if (before < need && incl >= need) {   // exactly one lane: the bin of the need-th largest
          int cum = before;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (cum + c[j] >= need) {
              sel_key = prefix | (static_cast<uint32_t>(255 - 8 * lane - j) << shift);
              sel_need = need - cum;
              break;
            }
            cum += c[j];
          }
        }
      }
      __syncthreads();
      prefix = sel_key;
      need = sel_need;
    }
    // keys above T are all taken; of the keys equal to T, the `need` lowest-indexed
    const uint32_t T = prefix;
    const int per = (len + kTopkThreads - 1) / kTopkThreads;
    const int i0 = min(len, static_cast<int>(threadIdx.x) * per), i1 = min(len, i0 + per);
    int eq = 0;
    for (int i = i0; i < i1; ++i) eq += order_key(sc[i]) == T;
    int eq_tot = 0, tot = 0;
    const int eq_base = block_excl_scan(eq, wsum, eq_tot);
    int cnt = 0;
    for (int i = i0, e = eq_base; i < i1; ++i) {
      const uint32_t k = order_key(sc[i]);
      cnt += (k > T || (k == T && e < need));
      e += k == T;
    }
    int o = block_excl_scan(cnt, wsum, tot);
    for (int i = i0, e = eq_base; i < i1; ++i) {
      const uint32_t k = order_key(sc[i]);
      if ((k > T || (k == T && e < need)) && o < nsel) list[o++] = i;   // o < nsel always holds
      e += k == T;
    }
  } else {
    for (int i = threadIdx.x; i < len; i += kTopkThreads) list[i] = i;
  }
  __syncthreads();

  // ---- 4. the listed V rows, weighted by their softmax probabilities ---------------
  // A V row is D/8 code words of 8 dims; a warp covers kTpw = 256/D rows at
  // a time (lane = slot * (D/8) + word).  Warp w takes list entries
  // kTpw*w + slot, then kTpw*kTopkWarps further on, eight rows per lane per
  // round with every load issued before any is used.  Each pair of dims is
  // restored as fp16(fmaf(c, scale, min)) and accumulated in fp32 (paired
  // FMA) in list order; the slots, then the warps, are summed in a fixed
  // order.
  {
    constexpr int kWords = D / 8;            // 32-bit code words per row
    constexpr int kTpw = 32 / kWords;        // rows a warp covers at once
    constexpr int kStep = kTpw * kTopkWarps;
    const int slotl = lane / kWords, word = lane % kWords;
    const int g = word / 8;                  // 64-group of this lane's dims
    float2 acc[4];                           // dims (0,4) (1,5) (2,6) (3,7) of the word
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u] = make_float2(0.0f, 0.0f);
    for (int j0 = warp * kTpw + slotl; j0 < nsel; j0 += 8 * kStep) {
      uint32_t cw[8];
      float mn[8], scl[8], e[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int j = j0 + r * kStep;
        if (j < nsel) {
          const int t = list[j];
          const int64_t slot = slot0 + t;
          cw[r] = *reinterpret_cast<const uint32_t*>(a.vc + slot * (D / 2) + 4 * word);
          mn[r] = a.vmin[slot * NG + g];
          scl[r] = a.vscale[slot * NG + g];
          e[r] = exp2f(sc[t] - M);
        } else {
          cw[r] = 0u;
          mn[r] = scl[r] = e[r] = 0.0f;
        }
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float2 s2 = make_float2(scl[r], scl[r]), m2 = make_float2(mn[r], mn[r]);
        const float2 e2 = make_float2(e[r], e[r]);
        const uint32_t y = cw[r] >> 8;
        const uint32_t h[4] = {restore_pair<false>(lop_mask_or(cw[r], kLoNib, kMagic), s2, m2),
                               restore_pair<true>(lop_mask_or(cw[r], kHiNib, kMagic), s2, m2),
                               restore_pair<false>(lop_mask_or(y, kLoNib, kMagic), s2, m2),
                               restore_pair<true>(lop_mask_or(y, kHiNib, kMagic), s2, m2)};
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] = q4::fma_f32x2(e2, unpack_h2(h[u]), acc[u]);
      }
    }
    // sum the row slots of the warp (lanes kWords apart), in slot order
#pragma unroll
    for (int o = kWords; o < 32; o <<= 1)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc[u].x += __shfl_xor_sync(0xffffffffu, acc[u].x, o);
        acc[u].y += __shfl_xor_sync(0xffffffffu, acc[u].y, o);
      }
    if (slotl == 0) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        red_o[warp][8 * word + u] = acc[u].x;
        red_o[warp][8 * word + u + 4] = acc[u].y;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < D) {
    float o = 0.0f;
#pragma unroll
    for (int w = 0; w < kTopkWarps; ++w) o += red_o[w][threadIdx.x];
    a.out[bi * a.ldo + h * D + threadIdx.x] = __float2half_rn(o / L);
  }
  if (idx_out != nullptr)
    for (int j = threadIdx.x; j < nsel; j += kTopkThreads) idx_out[static_cast<int64_t>(bh) * nsel + j] = list[j];
}

template <int D>
fg_status launch_topk(const fg_kv& kv, const void* q, int64_t ldq, const void* knew, const void* vnew,
                      int64_t ldnew, int64_t pos, int64_t keep, void* out, int64_t ldo, int32_t* idx,
                      cudaStream_t st) {
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  const int kMaxDyn = static_cast<int>(TopkLayout<D>::bytes(kTopkMaxLen, kTopkMaxLen));
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(decode_attn_topk_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDyn) !=
        cudaSuccess)
      return check_launch("decode_attn_topk smem attribute");
    attr_set[dev] = true;
  }
  DecodeArgs a = {};
  a.kc = kv.k_codes;
  a.vc = kv.v_codes;
  a.kmin = kv.k_mins;
  a.kscale = kv.k_scales;
  a.vmin = kv.v_mins;
  a.vscale = kv.v_scales;
  a.q = static_cast<const __half*>(q);
  a.ldq = ldq;
  a.knew = static_cast<const __half*>(knew);
  a.vnew = static_cast<const __half*>(vnew);
  a.ldnew = ldnew;
  a.pos = pos;
  a.out = static_cast<__half*>(out);
  a.ldo = ldo;
  a.heads = kv.heads;
  a.cap = kv.capacity;
  a.splits = 1;
  a.tps = 0;
  a.part = nullptr;
  a.err = device_error_word();
  if (!a.err) return fail(FG_ERR_CUDA, "device error word");
  a.wait_limit = wait_limit();
  const int64_t len = pos + 1, nsel = keep < len ? keep : len;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  Trace tr(KC_ATTN_TOPK, st);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(kv.b * kv.heads));
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = TopkLayout<D>::bytes(len, nsel);
  cfg.stream = st;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decode_attn_topk_kernel<D>, a, static_cast<int>(nsel), idx) != cudaSuccess)
    return check_launch("decode_attn_topk_kernel (launch)");
  return check_launch("decode_attn_topk_kernel");
}

}  // namespace

fg_status decode_attention_topk(const fg_kv& kv, const void* q, int64_t ldq, const void* knew, const void* vnew,
                                int64_t ldnew, int64_t pos, int64_t keep, void* out, int64_t ldo, int32_t* idx,
                                cudaStream_t st) {
  if (kv.b == 0) return FG_OK;
  if (kv.head_dim == 128) return launch_topk<128>(kv, q, ldq, knew, vnew, ldnew, pos, keep, out, ldo, idx, st);
  return launch_topk<64>(kv, q, ldq, knew, vnew, ldnew, pos, keep, out, ldo, idx, st);
}

fg_status check_decode_attention_topk(const fg_kv* kv, const void* q, int64_t ldq, int64_t pos, int64_t keep,
                                      const void* out, int64_t ldo, const int32_t* idx) {
  FG_TRY(check_decode_attention(kv, q, ldq, pos, out, ldo));
  if (keep < 1) return fail(FG_ERR_ARG, "keep %lld < 1", (long long)keep);
  if (kv->codec != FG_CODEC_Q4G64 || kv->dtype != FG_F16)
    return fail(FG_ERR_UNSUPPORTED, "top-K attention reads a 4-bit cache with fp16 activations");
  if (pos + 1 > kTopkMaxLen)
    return fail(FG_ERR_UNSUPPORTED, "top-K attention over %lld tokens (at most %lld)", (long long)(pos + 1),
                (long long)kTopkMaxLen);
  if (idx && !aligned(idx, 4)) return fail(FG_ERR_ALIGN, "idx needs 4-byte alignment");
  return FG_OK;
}

}  // namespace fg

extern "C" fg_status fg_decode_attention_topk(const fg_kv* kv, const void* q, int64_t ldq, int64_t pos,
                                              int64_t keep, void* out, int64_t ldo, int32_t* idx,
                                              cudaStream_t stream) {
  FG_TRY(fg::check_decode_attention_topk(kv, q, ldq, pos, keep, out, ldo, idx));
  if (kv->b == 0) return FG_OK;
  return fg::decode_attention_topk(*kv, q, ldq, nullptr, nullptr, 0, pos, keep, out, ldo, idx, stream);
}
