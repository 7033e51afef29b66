// Causal prefill attention on tcgen05 (FlexGen notes, "背景知识": x_Out =
// Softmax(x_Q x_K^T / sqrt(h1)) x_V per head, causal for generation;
// "5. 近似方法": K and V are read back from the 4-bit cache as FP16).
//
// Input: the layer's Q|K|V buffer [b*s][ld] (fp16) in which the K and V
// columns already hold the values the cache restores, fp16(fmaf(q, scale,
// min)) (written back by the K/V store), so that the attention reads
// exactly the cached values.  s is a multiple of 128.
//
// A persistent kernel: one CTA per SM takes items (sequence, head,
// 128-query tile) in units that pair a head's long and short query tiles,
// dealt round-robin so that a head's units run side by side (see PaItem),
// and runs each item flash-style over its 128-key tiles up to the diagonal:
//   * a TMA thread loads Q of an item into one of two buffers and the K, V
//     tiles into a two-stage ring that runs on across items (one tensor map
//     over the buffer, boxes of 64 columns x 128 rows, 128-byte swizzle:
//     K-major panels for Q and K, MN-major column blocks for V);
//   * one thread issues S = Q K^T (M = N = 128, K = head_dim) into tensor
//     memory and O += P V (K = 128 keys) into one of two O blocks (items
//     alternate), S of the next tile -- of this item or the next -- while
//     the softmax works on this one;
//   * four softmax warps (one query row per thread) read S with tcgen05.ld,
//     mask the diagonal tile, keep the running max and sum in base 2 and
//     write P (fp16) into shared memory in the swizzled K-major layout the
//     next MMA reads.  O is rescaled in tensor memory only when a row's max
//     grows by more than 2^8 (otherwise P is formed against the stale max,
//     which keeps it below 256 and the result the same up to rounding);
//   * after an item's last tile the softmax warps divide its O by the row
//     sums and store fp16, while the next item's S and P V proceed in the
//     other O block.
// The copy and MMA barriers count phases over the CTA's whole tile sequence.
// Every mbarrier wait is bounded; on timeout the CTA raises the library's
// device error word, lets its copies and MMAs finish and frees its tensor
// memory.
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <algorithm>

#include "fg_internal.cuh"
#include "tc_ptx.cuh"

namespace fg {

// defined in gemm_tc.cu
bool tc_make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

namespace {

using namespace tc;

constexpr int kTile = 128;          // queries per CTA, keys per tile
constexpr int kThreads = 192;       // warp 0: TMA, warp 1: MMA + TMEM, warps 2..5: softmax
constexpr int kSoftWarp0 = 2;
constexpr float kRescale = 8.0f;    // log2 growth of a row max that forces a rescale of O

struct PaParams {
  CUtensorMap map;      // the Q|K|V buffer, box {64, 128}
  __half* out;          // [b*s][ldo]
  int ldo;
  int s, heads, h1;
  int qtiles;           // s / 128
  int bh;               // b * heads
  int npairs;           // qtiles / 2: paired query tiles per head
  int pair_units;       // bh * npairs
  int units;            // pair_units + (bh if qtiles is odd)
  float scale_log2;     // log2(e) / sqrt(head_dim)
  unsigned int* err;
  uint32_t wait_limit;
};

template <int D>
struct PaSmem {
  static constexpr int kPanels = D / 64;          // 64-column panels of a head row
  static constexpr int kPanel = kTile * 128;      // 16 KiB: 128 rows x 128 bytes
  static constexpr int kQ = kPanels * kPanel;     // one Q buffer (two of them)
  static constexpr int kK = kPanels * kPanel;
  static constexpr int kV = kPanels * kPanel;     // MN-major: D/64 blocks of 128 keys x 64 dims
  static constexpr int kP = 2 * kPanel;           // 128 queries x 128 keys, two K-major panels
  static constexpr int kStage = kK + kV;
  static constexpr int kBytes = 1024 + 2 * kQ + 2 * kStage + kP + 256;
  static_assert(kBytes <= 232448, "shared memory of one CTA");
};

// 2^x on the special-function unit (relative error ~2^-22; P is rounded to
// fp16 right after, and 2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// acc + lo + hi of an fp16 pair, in fp32 (mixed-precision adds).
__device__ __forceinline__ float add_pair_f16(float acc, uint32_t h2) {
  float r;
  asm("{ .reg .f16 a, b; .reg .f32 t; mov.b32 {a, b}, %1; add.rn.f32.f16 t, a, %2; add.rn.f32.f16 %0, b, t; }"
      : "=f"(r)
      : "r"(h2), "f"(acc));
  return r;
}

// The work of a head (sequence bi, head h) is its query tiles qt = 0 ..
// qtiles-1, qt costing qt+1 key tiles.  Units pair tile qtiles-1-p with tile
// p (both cost qtiles+1 together); with an odd count the middle tile is a
// unit of its own.  Units run head by head, pairs before singles, dealt
// round-robin over the CTAs: every CTA gets the same work within one unit,
// and the two units of a head land on neighbouring CTAs in the same round,
// so that they read the head's K/V tiles from L2 rather than DRAM twice.
struct PaItem {
  int qt, bi, h;
};
// Items of CTA c (its units in order, a pair unit's longer tile first).
__device__ __forceinline__ int pa_pair_rounds(const PaParams& p, int c) {
  return c < p.pair_units ? (p.pair_units - c + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x) : 0;
}
__device__ __forceinline__ int pa_items(const PaParams& p, int c) {
  const int G = static_cast<int>(gridDim.x);
  const int rp = pa_pair_rounds(p, c);
  const int rall = c < p.units ? (p.units - c + G - 1) / G : 0;
  return 2 * rp + (rall - rp);
}
__device__ __forceinline__ PaItem pa_item(const PaParams& p, int c, int i) {
  const int G = static_cast<int>(gridDim.x);
  const int rp = pa_pair_rounds(p, c);
  int head, qt;
  if (i < 2 * rp) {
    const int u = c + (i >> 1) * G;
    head = u / p.npairs;
    const int pr = u - head * p.npairs;
    qt = (i & 1) ? pr : p.qtiles - 1 - pr;
  } else {
    const int u = c + (rp + (i - 2 * rp)) * G;
    head = u - p.pair_units;
    qt = p.qtiles >> 1;
  }
  PaItem it;
  it.qt = qt;
  it.bi = head / p.heads;
  it.h = head % p.heads;
  return it;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_attn_tc_kernel(const __grid_constant__ PaParams p) {
  using S = PaSmem<D>;
  constexpr uint32_t kIdescS = idesc_f16(128, 128, 0, 0);   // A = Q (K-major), B = K (K-major)
  constexpr uint32_t kIdescO = idesc_f16(128, D, 0, 1);     // A = P (K-major), B = V (MN-major)
  constexpr uint32_t kO = 128;                              // S: columns 0..127, O blocks from here
  constexpr uint32_t kTmemCols = kO + 2 * D <= 256 ? 256 : 512;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm;                          // two Q buffers
  uint8_t* sKV = sQ + 2 * S::kQ;             // two stages: [K panels][V blocks]
  uint8_t* sP = sKV + 2 * S::kStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + S::kP);
  uint64_t* qfull = bars;          // [2] Q of an item is in its buffer
  uint64_t* qfree = bars + 2;      // [2] the item's S MMAs have read it
  uint64_t* kvfull = bars + 4;     // [2]
  uint64_t* kvfree = bars + 6;     // [2] the PV MMA of the tile has read the stage
  uint64_t* sfull = bars + 8;      // S of the tile is in tensor memory
  uint64_t* sfree = bars + 9;      // four softmax warps have read S
  uint64_t* pfull = bars + 10;     // four softmax warps have written P
  uint64_t* odone = bars + 11;     // PV of the tile has completed
  uint64_t* ofree = bars + 12;     // [2] the softmax warps have stored the O block
  uint64_t* done = bars + 14;      // every MMA has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 15);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = static_cast<int>(blockIdx.x);
  const int nitems = pa_items(p, c);   // the host launches no CTA without work

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qfree[i], 1);
      mbar_init(&kvfull[i], 1);
      mbar_init(&kvfree[i], 1);
      mbar_init(&ofree[i], 4);
    }
    mbar_init(sfull, 1);
    mbar_init(sfree, 4);
    mbar_init(pfull, 4);
    mbar_init(odone, 1);
    mbar_init(done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  if (warp == 0 && lane == 0) tma_prefetch_desc(&p.map);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- TMA: per item Q, then K and V of each key tile ---------------------------
    if (lane == 0) {
      int q_issued = 0, g_issued = 0;
      bool ok = true;
      for (int i = 0; i < nitems && ok; ++i) {
        const PaItem it = pa_item(p, c, i);
        const int row0 = it.bi * p.s;
        const int qb = q_issued & 1;
        if (!mbar_wait(&qfree[qb], ((q_issued >> 1) & 1) ^ 1, p.wait_limit, abort_flag)) break;
        mbar_expect_tx(&qfull[qb], S::kQ);
        for (int pn = 0; pn < S::kPanels; ++pn)
          tma_load_2d(sQ + qb * S::kQ + pn * S::kPanel, &p.map, it.h * D + 64 * pn, row0 + it.qt * kTile, &qfull[qb]);
        ++q_issued;
        for (int j = 0; j <= it.qt; ++j) {
          const int st = g_issued & 1;
          if (!mbar_wait(&kvfree[st], ((g_issued >> 1) & 1) ^ 1, p.wait_limit, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* stage = sKV + st * S::kStage;
          mbar_expect_tx(&kvfull[st], S::kStage);
          for (int pn = 0; pn < S::kPanels; ++pn) {
            tma_load_2d(stage + pn * S::kPanel, &p.map, p.h1 + it.h * D + 64 * pn, row0 + j * kTile, &kvfull[st]);
            tma_load_2d(stage + S::kK + pn * S::kPanel, &p.map, 2 * p.h1 + it.h * D + 64 * pn, row0 + j * kTile,
                        &kvfull[st]);
          }
          ++g_issued;
        }
      }
      volatile int dummy = 0;   // nothing in flight at exit
      for (int u = (q_issued > 2 ? q_issued - 2 : 0); u < q_issued; ++u)
        mbar_wait(&qfull[u & 1], (u >> 1) & 1, kDrainLimit, &dummy);
      for (int u = (g_issued > 2 ? g_issued - 2 : 0); u < g_issued; ++u)
        mbar_wait(&kvfull[u & 1], (u >> 1) & 1, kDrainLimit, &dummy);
      if (*abort_flag) atomicOr(p.err, DEV_ERR_WAIT_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer, over the CTA's tile sequence -----------------------------------
    if (lane == 0) {
      const uint32_t p_addr = smem_u32(sP);
      // S of tile g (item n, Q buffer n & 1): needs K_g and a free S (tile
      // g-1's scores read); after an item's last S its Q buffer is released
      auto issue_s = [&](int g, int n, bool last) -> bool {
        const int st = g & 1;
        if (!mbar_wait(&kvfull[st], (g >> 1) & 1, p.wait_limit, abort_flag)) return false;
        if (g > 0 && !mbar_wait(sfree, (g - 1) & 1, p.wait_limit, abort_flag)) return false;
        tc_fence_after();
        const uint32_t q_addr = smem_u32(sQ + (n & 1) * S::kQ), k_addr = smem_u32(sKV + st * S::kStage);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * S::kPanel + (kk % 4) * 32;
          mma_f16(tmem, smem_desc_sw128(q_addr + off, 16, 1024), smem_desc_sw128(k_addr + off, 16, 1024), kIdescS,
                  kk > 0 ? 1u : 0u);
        }
        mma_commit(sfull);
        if (last) mma_commit(&qfree[n & 1]);
        return true;
      };
      bool ok = nitems > 0;
      int n = 0, j = 0, g = 0;   // item, its tile, the CTA's tile
      PaItem it = pa_item(p, c, 0);
      ok = ok && mbar_wait(&qfull[0], 0, p.wait_limit, abort_flag) && issue_s(0, 0, it.qt == 0);
      while (ok) {
        // the tile after g: the next of this item, or the first of the next item
        int nn = n, jn = j + 1;
        PaItem itn = it;
        if (jn > it.qt) {
          nn = n + 1;
          jn = 0;
          if (nn < nitems) itn = pa_item(p, c, nn);
        }
        const bool has_next = nn < nitems;
        if (has_next) {
          if (jn == 0 && !mbar_wait(&qfull[nn & 1], (nn >> 1) & 1, p.wait_limit, abort_flag)) {
            ok = false;
            break;
          }
          if (!issue_s(g + 1, nn, jn == itn.qt)) {
            ok = false;
            break;
          }
        }
        // O[n & 1] += P_g V_g; the block's first P V overwrites it, once the
        // softmax warps have stored the item that used it before
        if (!mbar_wait(pfull, g & 1, p.wait_limit, abort_flag) ||
            (j == 0 && !mbar_wait(&ofree[n & 1], ((n >> 1) & 1) ^ 1, p.wait_limit, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t v_addr = smem_u32(sKV + (g & 1) * S::kStage + S::kK);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          // A = P: K-major panels of 64 keys; B = V: 64-dim blocks 16 KiB apart
          // (leading byte offset), 8-key groups 1 KiB apart (stride)
          const uint64_t a = smem_desc_sw128(p_addr + (kk / 4) * S::kPanel + (kk % 4) * 32, 16, 1024);
          const uint64_t b = smem_desc_sw128(v_addr + kk * 2048, S::kPanel, 1024);
          mma_f16(tmem + kO + (n & 1) * D, a, b, kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&kvfree[g & 1]);   // K_g and V_g are read
        mma_commit(odone);
        if (!has_next) break;
        n = nn;
        j = jn;
        it = itn;
        ++g;
      }
      mma_commit(done);
      if (!ok) atomicOr(p.err, DEV_ERR_WAIT_TIMEOUT);
    }
    __syncwarp();
  } else if (warp >= kSoftWarp0) {
    // ---- softmax warps: query row r = 32 * (warp % 4) + lane of each item -------------
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
    uint8_t* prow = sP + r * 128;         // this row in each P panel
    bool ok = true;
    int g = 0, n = 0;
    for (; n < nitems && ok; ++n) {
      const PaItem it = pa_item(p, c, n);
      const uint32_t ob = kO + (n & 1) * D;
      const int qpos = it.qt * kTile + r;   // the query's position in its sequence (row r of the tile)
      float m = -INFINITY, l = 0.0f;
      for (int j = 0; j <= it.qt; ++j, ++g) {
        // tcgen05.ld/st are warp-collective: every branch around them is
        // taken by the whole warp
        if (ok) ok = mbar_wait(sfull, g & 1, p.wait_limit, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
        float sv[128];   // raw scores of the row (the scale is folded into the exponent below)
        if (ok) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t u[32];
            tmem_ld_32x32b_x32(trow + 32 * c, u);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) sv[32 * c + e] = __uint_as_float(u[e]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sfree);   // S may be overwritten by the next tile's scores
        // causal mask on the diagonal tile (the same for the whole warp): key
        // 128j + c is visible iff c <= r there
        if (j == it.qt) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > r) sv[c] = -INFINITY;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; ++c) mx = fmaxf(mx, sv[c]);
        mx *= p.scale_log2;   // in base-2 units, like m
        // P may be written once the previous tile's PV (of any item) has read
        // it; O may be rescaled only then too
        if (g > 0 && ok) ok = mbar_wait(odone, (g - 1) & 1, p.wait_limit, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
        if (j == 0) {
          m = mx;
        } else {
          // rows whose max grew by more than 2^8 take the new max and scale
          // their O by alpha; the other rows of the warp keep theirs (alpha 1)
          const bool grow = mx > m + kRescale;
          const float alpha = grow ? ex2_approx(m - mx) : 1.0f;
          if (grow) {
            l *= alpha;
            m = mx;
          }
          if (__any_sync(0xffffffffu, grow) && ok) {
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t u[32];
              tmem_ld_32x32b_x32(trow + ob + 32 * c, u);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
              tmem_st_32x32b_x32(trow + ob + 32 * c, u);
            }
            tmem_st_wait();
          }
        }
        // P = 2^(s * scale - m) in fp16, 8 keys (one 16-byte chunk) at a time,
        // into the swizzled K-major panels (chunk c8 of row r at c8 ^ (r % 8));
        // the row sum takes the fp16 weights the MMA multiplies
        const float negm = -m;
        float lsum = 0.0f;
#pragma unroll
        for (int c8 = 0; c8 < 16; ++c8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __half2 h2 = __floats2half2_rn(ex2_approx(fmaf(sv[8 * c8 + 2 * e], p.scale_log2, negm)),
                                                 ex2_approx(fmaf(sv[8 * c8 + 2 * e + 1], p.scale_log2, negm)));
            w[e] = *reinterpret_cast<const uint32_t*>(&h2);
            lsum = add_pair_f16(lsum, w[e]);
          }
          const int panel = c8 >> 3, chunk = c8 & 7;
          *reinterpret_cast<uint4*>(prow + panel * S::kPanel + ((chunk ^ (r & 7)) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
        l += lsum;
        fence_proxy_async_smem();   // P (generic writes) before the MMA reads it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pfull);
      }
      // ---- the item's O / l -> fp16, then its O block is free -----------------------
      if (ok) ok = mbar_wait(odone, (g - 1) & 1, p.wait_limit, abort_flag);
      ok = __all_sync(0xffffffffu, ok && !*abort_flag);
      tc_fence_after();
      if (ok) {
        const float inv = 1.0f / l;
        __half* dst = p.out + static_cast<size_t>(it.bi * p.s + qpos) * p.ldo + it.h * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t u[32];
          tmem_ld_32x32b_x32(trow + ob + 32 * c, u);
          tmem_ld_wait();
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __half2 h2 = __floats2half2_rn(__uint_as_float(u[8 * v + 2 * e]) * inv,
                                                   __uint_as_float(u[8 * v + 2 * e + 1]) * inv);
              w[e] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(dst + 32 * c + 8 * v) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ofree[n & 1]);
    }
  }
  // ---- teardown: every MMA done, then the tensor memory is freed ----------------------
  if (warp == 1 && lane == 0) {
    volatile int dummy = 0;
    mbar_wait(done, 0, kDrainLimit, &dummy);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
fg_status launch_pa(const void* qkv, int64_t ld, int64_t b, int64_t s, int32_t heads, void* out, int64_t ldo,
                    cudaStream_t st) {
  using S = PaSmem<D>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(prefill_attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes) !=
        cudaSuccess)
      return check_launch("prefill_attn_tc smem attribute");
    attr_set[dev] = true;
  }
  PaParams p;
  memset(&p, 0, sizeof(p));
  if (!tc_make_map(&p.map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qkv, static_cast<uint64_t>(ld), static_cast<uint64_t>(b * s),
                   static_cast<uint64_t>(ld) * 2, 64, kTile, CU_TENSOR_MAP_SWIZZLE_128B))
    return fail(FG_ERR_CUDA, "tensor map for the Q|K|V buffer");
  p.out = static_cast<__half*>(out);
  p.ldo = static_cast<int>(ldo);
  p.s = static_cast<int>(s);
  p.heads = heads;
  p.h1 = heads * D;
  p.qtiles = static_cast<int>(s / kTile);
  p.bh = static_cast<int>(b * heads);
  p.npairs = p.qtiles / 2;
  p.pair_units = p.bh * p.npairs;
  p.units = p.pair_units + (p.qtiles % 2 ? p.bh : 0);
  p.scale_log2 = static_cast<float>(1.4426950408889634074 / sqrt(static_cast<double>(D)));
  p.err = device_error_word();
  if (!p.err) return fail(FG_ERR_CUDA, "device error word");
  p.wait_limit = wait_limit();
  Trace tr(KC_ATTN_PREFILL, st);
  // persistent: one CTA per SM (the shared memory admits no second one),
  // and no more CTAs than units
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(p.units, num_sms()));
  prefill_attn_tc_kernel<D><<<grid, kThreads, S::kBytes, st>>>(p);
  return check_launch("prefill_attn_tc_kernel");
}

}  // namespace

bool prefill_attention_tc_supported(int64_t s, int32_t head_dim, fg_dtype dt) {
  return dt == FG_F16 && s >= kTile && s % kTile == 0 && (head_dim == 64 || head_dim == 128);
}

fg_status prefill_attention_tc(const void* qkv, int64_t ld, int64_t b, int64_t s, int32_t heads, int32_t head_dim,
                               void* out, int64_t ldo, cudaStream_t st) {
  if (b == 0 || s == 0) return FG_OK;
  if (!aligned(qkv, 16) || (ld * 2) % 16 || !aligned(out, 16) || ldo % 8)
    return fail(FG_ERR_ALIGN, "prefill attention: 16-byte aligned buffers and rows");
  if (head_dim == 128) return launch_pa<128>(qkv, ld, b, s, heads, out, ldo, st);
  return launch_pa<64>(qkv, ld, b, s, heads, out, ldo, st);
}

}  // namespace fg
