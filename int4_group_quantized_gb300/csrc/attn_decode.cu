// Decode attention over the 4-bit KV cache with the new token's K/V appended
// in the same launch (FlexGen notes, "背景知识": x_K <- Concat(x_K, t w_K),
// x_V <- Concat(x_V, t w_V), t_Out = Softmax(t_Q x_K^T / sqrt(h1)) x_V;
// "5. 近似方法": K/V stored in 4-bit groups of 64 along the hidden dimension).
//
// The path is HBM-bound (one query per (sequence, head) against ~0.6 bytes
// per cached value), so the design goal is to convert codes with as few
// instructions as possible.  Codes never become full fp16 values:
//   * a lop3 with 0x6400 in the exponent turns a nibble c into the exact
//     fp16 number 1024 + c (or 1024 + 16c for the upper nibble of a byte);
//   * the legacy warp-level tensor-core MMA (m16n8k16, fp32 accumulate)
//     forms the dot products on these biased integers; the bias is removed
//     once per group: sum_j q_j (1024 + c_j) = sum_j q_j c_j + 1024 sum_j q_j;
//   * the per-token (min, scale) pair is applied to the group's integer dot
//     product: k.q = scale * sum_j c_j q_j + min * sum_j q_j, and for the
//     values sum_t p_t (c_t scale_t + min_t) = sum_t (p_t scale_t) c_t +
//     sum_t p_t min_t.
// That is ~0.7 integer instructions per cached element; the MMAs carry the
// multiply-adds.
//
// One CTA (4 warps) per (sequence, head, token split).  Each warp walks its
// tokens 16 at a time with an online softmax in base 2 (the fp32 scores are
// scaled by log2(e)/sqrt(d)); warps, then splits, are merged with the usual
// max/sum rescaling.
#include <math.h>

#include "attn_dev.cuh"
#include "fg_internal.cuh"
#include "tc_ptx.cuh"

namespace fg {
namespace {

using namespace attn;

// Registers holding one 16-token block of the cache as a lane needs it.
template <int NG>
struct KVBlock {
  uint2 kw[2][NG];      // K codes of tokens gq, gq+8 (8 bytes per group)
  uint32_t vw[4][NG];   // V codes of tokens 2tig, 2tig+1, 2tig+8, 2tig+9 (4 bytes per group)
  float ksc[2][NG], kmn[2][NG], vsc[2][NG], vmn[2][NG];   // (scale, min) of tokens gq, gq+8
};

// One 16-token block of the cache (tokens tb .. tb+15, valid below t1) into
// a warp's running softmax state and output accumulators.
template <int D>
struct WarpState {
  static constexpr int NG = D / 64;
  static constexpr int NT = D / 16;
  uint32_t qb[NG][4][2];   // q as B fragments (biased-integer form, see the header)
  float bias[NG], qsum[NG];
  float run_m, run_l;
  float ps[NG], cmn[NG];
  float acc[NT][4];
};

template <int D>
__device__ __forceinline__ void process_block(WarpState<D>& W, int64_t tb, int64_t t1, const KVBlock<D / 64>& B,
                                              int gq, int tig) {
  constexpr int NG = D / 64;
  constexpr int NT = D / 16;
  auto& run_m = W.run_m;
  auto& run_l = W.run_l;
  auto& ps = W.ps;
  auto& cmn = W.cmn;
  auto& acc = W.acc;
    const bool kval[2] = {tb + gq < t1, tb + gq + 8 < t1};
    const auto& kw = B.kw;
    const auto& vw = B.vw;
    const auto& ksc = B.ksc;
    const auto& kmn = B.kmn;
    const auto& vsc = B.vsc;
    const auto& vmn = B.vmn;

    // scores (base 2) of tokens gq and gq+8
    float sc0, sc1;
    block_scores<NG>(W, kw, ksc, kmn, sc0, sc1);
    constexpr float kQs = score_scale_log2<D>();
    sc0 *= kQs;
    sc1 *= kQs;
    if (!kval[0]) sc0 = -INFINITY;
    if (!kval[1]) sc1 = -INFINITY;

    // online softmax over the block
    float m = fmaxf(sc0, sc1);
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
    const float new_m = fmaxf(run_m, m);
    const float alpha = exp2f(run_m - new_m);
    const float p0 = exp2f(sc0 - new_m), p1 = exp2f(sc1 - new_m);
    // run_l, ps and cmn are kept per lane (this lane's tokens; alpha is the
    // same in every lane) and reduced across the warp once, after the last block
    run_l = run_l * alpha + (p0 + p1);
    run_m = new_m;

    // value weights p*scale per group, as B fragments for tokens
    // (2tig, 2tig+1 | 2tig+8, 2tig+9), and the min term sum p*min
    uint32_t vb[NG][2];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const float w0 = p0 * vsc[0][g], w1 = p1 * vsc[1][g];
      const float a0 = __shfl_sync(0xffffffffu, w0, 8 * tig);
      const float a1 = __shfl_sync(0xffffffffu, w0, 8 * tig + 4);
      const float a8 = __shfl_sync(0xffffffffu, w1, 8 * tig);
      const float a9 = __shfl_sync(0xffffffffu, w1, 8 * tig + 4);
      vb[g][0] = pack_h2(a0, a1);
      vb[g][1] = pack_h2(a8, a9);
      const float2 u = unpack_h2(vb[g][0]), v = unpack_h2(vb[g][1]);
      ps[g] = ps[g] * alpha + (u.x + u.y + v.x + v.y);   // the fp16 weights the MMA multiplies
      cmn[g] = cmn[g] * alpha + (p0 * vmn[0][g] + p1 * vmn[1][g]);
    }

    // O^T[dim] += sum_t V^T[dim][t] * (p scale)[t]; tile i covers dims
    // 64*(i/4) + 8*gq + 2*(i%4) (+1 for the upper row, scaled x16)
    // the running max is the same in every lane, and after the first blocks
    // it rarely moves: the rescale is skipped when it did not
    if (alpha != 1.0f) {
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        acc[i][0] *= alpha;
        acc[i][1] *= alpha;
        acc[i][2] *= alpha;
        acc[i][3] *= alpha;
      }
    }
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const int g = i / 4, ii = i % 4;
      const uint32_t sel = static_cast<uint32_t>(ii) | (static_cast<uint32_t>(ii + 4) << 8);
      const uint32_t x01 = __byte_perm(vw[0][g], vw[1][g], sel);
      const uint32_t x89 = __byte_perm(vw[2][g], vw[3][g], sel);
      mma16816(acc[i], lop_mask_or(x01, kLoNib, kMagic), lop_mask_or(x01, kHiNib, kMagic),
               lop_mask_or(x89, kLoNib, kMagic), lop_mask_or(x89, kHiNib, kMagic), vb[g][0], vb[g][1]);
    }
}

// Merge the 4 attention warps of a CTA (shared red_*), then write the result
// (one split) or this split's partial (several).  Every thread of the CTA
// calls it (it holds a CTA barrier); only attention warps stash.
template <int D>
__device__ __forceinline__ void merge_warps(const WarpState<D>& W, float* red_m, float* red_l, float (*red_o)[D],
                                            const DecodeArgs& a, int64_t bi, int h, int bh, int sp, int warp,
                                            int lane, int gq, int tig, bool stash = true) {
  constexpr int NT = D / 16;
  const auto& acc = W.acc;
  const auto& ps = W.ps;
  const auto& cmn = W.cmn;
  const float run_m = W.run_m, run_l = W.run_l;
  if (stash && tig == 0) {
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const int g = i / 4, ii = i % 4;
      const int dim = 64 * g + 8 * gq + 2 * ii;
      red_o[warp][dim] = (acc[i][0] - 1024.0f * ps[g]) + cmn[g];
      red_o[warp][dim + 1] = (acc[i][2] - 1024.0f * ps[g]) * 0.0625f + cmn[g];
    }
  }
  if (stash && lane == 0) {
    red_m[warp] = run_m;
    red_l[warp] = run_l;
  }
  __syncthreads();
  if (threadIdx.x < D) {
    const int dim = threadIdx.x;
    float M = fmaxf(fmaxf(red_m[0], red_m[1]), fmaxf(red_m[2], red_m[3]));
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float f = red_m[w] == -INFINITY ? 0.0f : exp2f(red_m[w] - M);
      L += f * red_l[w];
      O += f * red_o[w][dim];
    }
    if (a.splits == 1) {
      a.out[bi * a.ldo + h * D + dim] = __float2half_rn(O / L);
    } else {
      float* p = a.part + (static_cast<int64_t>(bh) * a.splits + sp) * (D + 2);
      p[dim] = O;
      if (dim == 0) {
        p[D] = M;
        p[D + 1] = L;
      }
    }
  }
}

// Each warp stages its own 16-token blocks in shared memory, kWStages deep,
// with asynchronous copies (per-thread groups, no CTA barrier): the K and V
// codes of the block's rows in 16-byte pieces, and each row's (scale, min)
// pairs.  The warp reads a block from shared memory right before it uses
// it, so no registers hold blocks in flight.
constexpr int kWStages = 3;

template <int D>
struct WarpStage {
  static constexpr int C = D / 2;            // code bytes of a row
  static constexpr int NG = D / 64;
  static constexpr int kMetaArr = 16 * NG * 4;   // one (scale or min) array of a block
  static constexpr int kK = 0, kV = 16 * C;
  static constexpr int kKs = 32 * C, kKm = kKs + kMetaArr, kVs = kKm + kMetaArr, kVm = kVs + kMetaArr;
  static constexpr int kBytes = kVm + kMetaArr;
};

template <int D>
__global__ void __launch_bounds__(128, 4) decode_attn_mma_kernel(const DecodeArgs a) {
  constexpr int NG = D / 64;   // 64-groups per head row
  constexpr int NT = D / 16;   // m16 tiles of value dims
  using WS = WarpStage<D>;
  __shared__ float red_m[4], red_l[4];
  __shared__ float red_o[4][D];
  __shared__ __align__(16) uint8_t wsm[4][kWStages][WS::kBytes];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gq = lane >> 2, tig = lane & 3;
  const int bh = blockIdx.x / a.splits, sp = blockIdx.x % a.splits;
  const int64_t bi = bh / a.heads;
  const int h = bh % a.heads;
  const int64_t len = a.pos + 1;
  const int64_t t0 = static_cast<int64_t>(sp) * a.tps;
  const int64_t t1 = min(len, t0 + a.tps);
  const int64_t slot0 = static_cast<int64_t>(bh) * a.cap;

  // launched with programmatic stream serialization: the next kernel may be
  // scheduled now; q, the new K/V and the cache are read after the previous
  // kernel has completed
  tc::griddep_launch();
  tc::griddep_wait();

  // ---- Concat: quantize the new token's K and V into slot pos -----------------
  if (a.knew != nullptr && a.pos >= t0 && a.pos < t1) {
    if (warp == 0) {
      append_token<D>(a, slot0, bi, h, lane);
      tc::fence_proxy_async_global();   // the new row, then the asynchronous copies that read it
    }
    __syncthreads();
  }

  // ---- q as B fragments ---------------------------------------------------------
  WarpState<D> W;
  setup_q<D>(W, a.q + bi * a.ldq + h * D, tig);

  // ---- this warp's tokens -------------------------------------------------------
  const int nblk = static_cast<int>((t1 - t0 + 15) / 16);
  const int wb0 = warp * nblk / 4, wb1 = (warp + 1) * nblk / 4;
  auto& run_m = W.run_m;
  auto& run_l = W.run_l;
  auto& ps = W.ps;
  auto& cmn = W.cmn;
  auto& acc = W.acc;
  run_m = -INFINITY;
  run_l = 0.0f;
#pragma unroll
  for (int g = 0; g < NG; ++g) ps[g] = cmn[g] = 0.0f;
#pragma unroll
  for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;

  // block blk of this CTA's tokens into this warp's stage st.  The pieces a
  // lane copies sit at the same offsets in every block (rows are contiguous):
  // lane l copies 16-byte pieces l, l + 32, ... of the K and V codes and
  // floats l, l + 32, ... of the four (scale, min) arrays' NG * 16.
  constexpr int kPieces = 16 * WS::C / 16;                    // 16-byte pieces of a block's codes
  constexpr int kMetaPer = (64 * NG + 31) / 32;               // pair floats a lane copies
  const uint8_t* kc_l = a.kc + (slot0 + t0) * WS::C + 16 * lane;
  const uint8_t* vc_l = a.vc + (slot0 + t0) * WS::C + 16 * lane;
  const float* meta_l[kMetaPer];
  int meta_dst[kMetaPer], meta_row[kMetaPer];
#pragma unroll
  for (int u = 0; u < kMetaPer; ++u) {
    const int e = lane + 32 * u, arr = e / (16 * NG), f = e % (16 * NG);
    const float* base = arr == 0 ? a.kscale : arr == 1 ? a.kmin : arr == 2 ? a.vscale : a.vmin;
    meta_l[u] = base + (slot0 + t0) * NG + f;
    meta_dst[u] = WS::kKs + arr * WS::kMetaArr + f * 4;
    meta_row[u] = f / NG;
  }
  auto issue = [&](int blk, int st) {
    const int64_t tb = t0 + static_cast<int64_t>(blk) * 16;
    const int nrow = static_cast<int>(min(static_cast<int64_t>(16), t1 - tb));   // valid rows of the block
    uint8_t* s = wsm[warp][st];
    const int64_t cb = static_cast<int64_t>(blk) * 16 * WS::C;
#pragma unroll
    for (int pc = lane, u = 0; u < (kPieces + 31) / 32; pc += 32, ++u) {
      if (pc < kPieces && pc / (WS::C / 16) < nrow) {
        tc::cp_async16(s + WS::kK + 16 * pc, kc_l + cb + 512 * u);
        tc::cp_async16(s + WS::kV + 16 * pc, vc_l + cb + 512 * u);
      }
    }
    const int64_t mb = static_cast<int64_t>(blk) * 16 * NG;
#pragma unroll
    for (int u = 0; u < kMetaPer; ++u)
      if (meta_row[u] < nrow) tc::cp_async4(s + meta_dst[u], meta_l[u] + mb);
    tc::cp_async_commit();
  };

  // block blk from stage st into registers, as process_block takes it (rows
  // past t1 read as zero)
  auto read = [&](int blk, int st, KVBlock<NG>& B) {
    const int64_t tb = t0 + static_cast<int64_t>(blk) * 16;
    const uint8_t* s = wsm[warp][st];
    if (tb + 16 <= t1) {   // a full block: no row to mask
      const float* ks = reinterpret_cast<const float*>(s + WS::kKs);
      const float* km = reinterpret_cast<const float*>(s + WS::kKm);
      const float* vs = reinterpret_cast<const float*>(s + WS::kVs);
      const float* vm = reinterpret_cast<const float*>(s + WS::kVm);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = gq + 8 * r;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          B.kw[r][g] = *reinterpret_cast<const uint2*>(s + WS::kK + row * WS::C + g * 32 + 8 * tig);
          B.ksc[r][g] = ks[row * NG + g];
          B.kmn[r][g] = km[row * NG + g];
          B.vsc[r][g] = vs[row * NG + g];
          B.vmn[r][g] = vm[row * NG + g];
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = 2 * tig + (r & 1) + 8 * (r >> 1);
#pragma unroll
        for (int g = 0; g < NG; ++g)
          B.vw[r][g] = *reinterpret_cast<const uint32_t*>(s + WS::kV + row * WS::C + g * 32 + 4 * gq);
      }
      return;
    }
    const float* ks = reinterpret_cast<const float*>(s + WS::kKs);
    const float* km = reinterpret_cast<const float*>(s + WS::kKm);
    const float* vs = reinterpret_cast<const float*>(s + WS::kVs);
    const float* vm = reinterpret_cast<const float*>(s + WS::kVm);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = gq + 8 * r;
      const bool v = tb + row < t1;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        B.kw[r][g] = v ? *reinterpret_cast<const uint2*>(s + WS::kK + row * WS::C + g * 32 + 8 * tig)
                       : make_uint2(0u, 0u);
        B.ksc[r][g] = v ? ks[row * NG + g] : 0.0f;
        B.kmn[r][g] = v ? km[row * NG + g] : 0.0f;
        B.vsc[r][g] = v ? vs[row * NG + g] : 0.0f;
        B.vmn[r][g] = v ? vm[row * NG + g] : 0.0f;
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = 2 * tig + (r & 1) + 8 * (r >> 1);
      const bool v = tb + row < t1;
#pragma unroll
      for (int g = 0; g < NG; ++g)
        B.vw[r][g] = v ? *reinterpret_cast<const uint32_t*>(s + WS::kV + row * WS::C + g * 32 + 4 * gq) : 0u;
    }
  };

  // the pipeline: blocks wb0.. in stages j % kWStages, kWStages - 1 ahead
#pragma unroll
  for (int i = 0; i < kWStages - 1; ++i) {
    if (wb0 + i < wb1) issue(wb0 + i, i);
    else tc::cp_async_commit();
  }
  for (int blk = wb0; blk < wb1; ++blk) {
    const int j = blk - wb0;
    // stage (j + kWStages - 1) % kWStages was read in iteration j - 1, which
    // ended with a warp barrier
    if (blk + kWStages - 1 < wb1) issue(blk + kWStages - 1, (j + kWStages - 1) % kWStages);
    else tc::cp_async_commit();
    tc::cp_async_wait<kWStages - 1>();   // this lane's copies of block blk have landed
    __syncwarp();                        // and every lane's
    KVBlock<NG> B;
    read(blk, j % kWStages, B);
    process_block<D>(W, t0 + static_cast<int64_t>(blk) * 16, t1, B, gq, tig);
    __syncwarp();                        // stage j % kWStages is read
  }

  // the per-lane sums over this warp's tokens: run_l and cmn over the rows gq
  // (lanes 4 apart), ps over the token pairs of tig (lanes 1 apart)
  W.run_l += __shfl_xor_sync(0xffffffffu, W.run_l, 4);
  W.run_l += __shfl_xor_sync(0xffffffffu, W.run_l, 8);
  W.run_l += __shfl_xor_sync(0xffffffffu, W.run_l, 16);
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    W.ps[g] += __shfl_xor_sync(0xffffffffu, W.ps[g], 1);
    W.ps[g] += __shfl_xor_sync(0xffffffffu, W.ps[g], 2);
    W.cmn[g] += __shfl_xor_sync(0xffffffffu, W.cmn[g], 4);
    W.cmn[g] += __shfl_xor_sync(0xffffffffu, W.cmn[g], 8);
    W.cmn[g] += __shfl_xor_sync(0xffffffffu, W.cmn[g], 16);
  }
  merge_warps<D>(W, red_m, red_l, red_o, a, bi, h, bh, sp, warp, lane, gq, tig);
}

// Merge the token splits of each (sequence, head).
template <int D>
__global__ void decode_attn_combine_kernel(const float* __restrict__ part, int splits, int heads,
                                           __half* __restrict__ out, int64_t ldo) {
  tc::griddep_launch();
  tc::griddep_wait();
  const int bh = blockIdx.x, dim = threadIdx.x;
  const float* p = part + static_cast<int64_t>(bh) * splits * (D + 2);
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, p[s * (D + 2) + D]);
  float L = 0.0f, O = 0.0f;
  for (int s = 0; s < splits; ++s) {
    const float m = p[s * (D + 2) + D];
    const float f = m == -INFINITY ? 0.0f : exp2f(m - M);
    L += f * p[s * (D + 2) + D + 1];
    O += f * p[s * (D + 2) + dim];
  }
  out[static_cast<int64_t>(bh / heads) * ldo + (bh % heads) * D + dim] = __float2half_rn(O / L);
}

// Token splits per (sequence, head): enough CTAs for ~6 per SM, at least 64
// tokens each.  Depends on the shape only.
int attn_splits(int64_t bh, int64_t len) {
  const int64_t target = 148 * 6;
  int64_t s = (target + bh - 1) / bh;
  const int64_t by_len = (len + 63) / 64;
  if (s > by_len) s = by_len;
  if (s > 32) s = 32;
  return static_cast<int>(s < 1 ? 1 : s);
}

template <int D>
fg_status launch_mma(const fg_kv& kv, const void* q, int64_t ldq, const void* knew, const void* vnew,
                     int64_t ldnew, int64_t b, int64_t pos, void* out, int64_t ldo, void* ws,
                     size_t ws_bytes, cudaStream_t st) {
  DecodeArgs a;
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
  const int64_t bh = b * kv.heads, len = pos + 1;
  const int want = attn_splits(bh, len);
  a.tps = static_cast<int>(((len + want - 1) / want + 15) / 16 * 16);
  a.splits = static_cast<int>((len + a.tps - 1) / a.tps);
  a.part = nullptr;
  if (a.splits > 1) {
    const size_t need = static_cast<size_t>(bh) * a.splits * (D + 2) * sizeof(float);
    if (!ws || ws_bytes < need) return fail(FG_ERR_WORKSPACE, "attention split partials need %zu bytes", need);
    a.part = static_cast<float*>(ws);
  }
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  {
    Trace tr(KC_ATTN_DECODE, st);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(bh * a.splits));
    cfg.blockDim = dim3(128);
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_attn_mma_kernel<D>, a) != cudaSuccess)
      return check_launch("decode_attn_mma_kernel (launch)");
  }
  {
    const fg_status s = check_launch("decode_attn_mma_kernel");
    if (s != FG_OK) return s;
  }
  if (a.splits > 1) {
    Trace tr(KC_ATTN_COMBINE, st);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(bh));
    cfg.blockDim = dim3(D);
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_attn_combine_kernel<D>, static_cast<const float*>(a.part), a.splits,
                           static_cast<int>(kv.heads), a.out, ldo) != cudaSuccess)
      return check_launch("decode_attn_combine_kernel (launch)");
    return check_launch("decode_attn_combine_kernel");
  }
  return FG_OK;
}

}  // namespace

size_t decode_attention_workspace_bytes(int64_t b, int32_t heads, int32_t head_dim, int64_t capacity) {
  const int64_t bh = b * heads;
  const int s = attn_splits(bh, capacity);
  return s > 1 ? static_cast<size_t>(bh) * s * (head_dim + 2) * sizeof(float) : 0;
}

fg_status decode_attention(const fg_kv& kv, const void* q, int64_t ldq, const void* knew,
                           const void* vnew, int64_t ldnew, int64_t b, int64_t pos, void* out,
                           int64_t ldo, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (b == 0) return FG_OK;
  if (kv.codec == FG_CODEC_Q4G64 && kv.dtype == FG_F16) {
    if (kv.head_dim == 128)
      return launch_mma<128>(kv, q, ldq, knew, vnew, ldnew, b, pos, out, ldo, ws, ws_bytes, st);
    if (kv.head_dim == 64)
      return launch_mma<64>(kv, q, ldq, knew, vnew, ldnew, b, pos, out, ldo, ws, ws_bytes, st);
  }
  // fp32 activations or an uncompressed cache: append, then CUDA-core attention
  if (knew) {
    fg_status s = kv_store(kv, knew, vnew, ldnew, b, 1, pos, st);
    if (s != FG_OK) return s;
  }
  return decode_attention_simt(kv, q, ldq, b, pos, out, ldo, st);
}

}  // namespace fg

// ---------------------------------------------------------------------------
// Decode attention for callers that cannot allocate device memory.
//
// The split-over-tokens partial results normally live in a workspace the
// caller allocates.  This entry point uses instead a fixed array compiled
// into the library, which every GPU that loads libfg.so holds until the
// process exits.  Its device address is looked up once per device (with
// that device current) by the first call on that device and then cached
// for the life of the process; make that first call before any stream
// capture and before any region in which allocations are forbidden (with
// lazy module loading, that first call is also what loads this code onto
// the device).  A device reset or a destroyed primary context invalidates
// the cached address.  Every call shares the array: calls whose kernels
// overlap on the GPU race on it.  Nothing in it needs to start at zero
// (each split writes its partial before the merge reads it).
// ---------------------------------------------------------------------------
#include <mutex>

// The split rule above asks for b*H*splits*(d+2)*4 bytes.  Splits happen only
// while b*H < 888; with head_dim 128 the largest need is at b*H = 887 with two
// splits, 1774*130*4 = 922,480 bytes (head_dim 64: less), so 1 MiB covers
// every cache (a host-side sweep in the tests checks it).
static constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;   // 1 MiB
static __device__ __align__(256) unsigned char g_decode_attn_scratch[kNoAllocScratchBytes];

static fg_status noalloc_scratch(void** ptr) {
  static std::mutex mu;
  static void* cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fg::fail(FG_ERR_CUDA, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_attn_scratch);
    if (e != cudaSuccess) return fg::fail(FG_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    cache[dev] = p;
  }
  *ptr = cache[dev];
  return FG_OK;
}

extern "C" fg_status fg_decode_attention_noalloc(const fg_kv* kv, const void* q, int64_t ldq, int64_t pos,
                                                 void* out, int64_t ldo, cudaStream_t stream) {
  // every host-side check first, so that bad arguments never reach a CUDA call
  const fg_status c = fg::check_decode_attention(kv, q, ldq, pos, out, ldo);
  if (c != FG_OK) return c;
  const size_t need = fg_decode_attention_workspace_bytes(kv);
  if (need > kNoAllocScratchBytes)
    return fg::fail(FG_ERR_WORKSPACE,
                    "this cache needs %zu bytes of split scratch; the built-in array holds %zu "
                    "(use fg_decode_attention with a caller workspace)",
                    need, kNoAllocScratchBytes);
  if (kv->b == 0) return FG_OK;
  void* scratch = nullptr;
  const fg_status s = noalloc_scratch(&scratch);
  if (s != FG_OK) return s;
  return fg_decode_attention(kv, q, ldq, pos, out, ldo, scratch, kNoAllocScratchBytes, stream);
}
