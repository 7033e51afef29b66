// Tensor-core products on sm_103a: Y = epilogue(X . W) with tcgen05.mma
// (fp16 operands, fp32 accumulator in TMEM), operands staged by TMA.
//
// FlexGen notes, "背景知识": the layer's products x w_Q, x w_K, x w_V, (..) w_O
// + x, relu(x_Out w_1), (..) w_2 + x_Out; "5. 近似方法": weights stored in
// 4-bit groups of 64 along the output channel and converted back to FP16
// before compute.
//
// The weight operand B is fp16 [K][N] row-major (MN-major): for the prefill
// products (b*s rows) the layer's 4-bit weights were converted back to fp16
// once per layer, and every tile of them then feeds many rows.  A = X tiles
// [128 rows][64 k] (K-major, 128-byte swizzle) and B tiles come by TMA; rows
// past M are zero-filled by the TMA unit.
//
// Warp roles (256 threads): warp 0 issues TMA; warp 1 owns TMEM and one of
// its lanes issues the MMAs; then all eight warps drain the accumulator in
// the epilogue (warp w: TMEM lanes 32(w%4).., half of the tile's columns).
// Every wait is bounded: on timeout the CTA raises the library's device
// error word and leaves.

#include <cudaTypedefs.h>
#include <string.h>

#include "fg_internal.cuh"
#include "tc_ptx.cuh"

namespace fg {
namespace {

using namespace tc;

constexpr int BK = 64;             // k per pipeline stage (one 128-byte swizzle row of fp16)
constexpr int kThreads = 256;
constexpr int BN = 256;            // columns of a CTA tile

struct TcParams {
  CUtensorMap mapA;
  CUtensorMap mapB[3];      // fp16 W [K][N_seg], box {64, 64}
  int seg_n0[4];            // segment column offsets, seg_n0[nseg] = N
  int nseg;
  int M, N, K;
  int m_tiles, n_tiles, splits, ktiles_per_split;
  int group_n;              // raster: CTAs sweep M inside groups of group_n column tiles
  __half* Y;
  int ldy;
  const __half* R;
  int ldr;
  int relu;
  float* partial;           // splits > 1: [splits][M][N]
  unsigned int* err;
  uint32_t wait_limit;      // polls of a bounded wait (fg_set_wait_limit)
};

template <int MT>
struct Smem {
  static constexpr int kA = MT * 128 * BK * 2;           // bytes of A per stage
  static constexpr int kB = BK * BN * 2;                 // fp16 B tile
  static constexpr int kTx = kA + kB;                    // TMA bytes per stage
  static constexpr int kStage = (kTx + 1023) / 1024 * 1024;
  static constexpr int kBudget = 220 * 1024;
  static constexpr int kStages = kBudget / kStage > 8 ? 8 : kBudget / kStage;
  static constexpr int kTotal = 1024 /*align slack*/ + kStages * kStage + 256;
  static_assert(kStages >= 2, "pipeline needs two stages");
  static_assert(kA % 1024 == 0 && kB % 1024 == 0, "swizzle atoms need 1 KiB alignment");
};

__device__ __forceinline__ void raise(const TcParams& p) { atomicOr(p.err, DEV_ERR_WAIT_TIMEOUT); }

template <int MT>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ TcParams p) {
  using S = Smem<MT>;
  constexpr int STAGES = S::kStages;
  constexpr uint32_t kTmemCols = MT * BN;   // 128, 256 or 512
  constexpr uint32_t kIdesc = idesc_f16(128, BN, 0, 1);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  uint8_t* tail = smem + STAGES * S::kStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(tail);
  uint64_t* empty = full + STAGES;
  uint64_t* done = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- tile coordinates -------------------------------------------------------
  int tile = blockIdx.x;
  const int split = tile % p.splits;
  tile /= p.splits;
  int mt_idx, nt_idx;
  {
    // groups of group_n column tiles; inside a group, consecutive CTAs walk
    // the column tiles first so an A panel is reused from L2
    const int per_group = p.group_n * p.m_tiles;
    const int g = tile / per_group;
    const int in = tile % per_group;
    const int gw = min(p.group_n, p.n_tiles - g * p.group_n);
    nt_idx = g * p.group_n + in % gw;
    mt_idx = in / gw;
  }
  const int m0 = mt_idx * MT * 128;
  const int n0 = nt_idx * BN;
  int seg = 0;
  while (seg + 1 < p.nseg && n0 >= p.seg_n0[seg + 1]) ++seg;
  const int nl = n0 - p.seg_n0[seg];
  const int kt0 = split * p.ktiles_per_split;
  const int kt1 = min(kt0 + p.ktiles_per_split, p.K / BK);
  const int nk = kt1 - kt0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);   // the MMA commit
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.mapA);
    tma_prefetch_desc(&p.mapB[seg]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---- TMA producer -----------------------------------------------------------
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(&empty[s], ((i / STAGES) & 1) ^ 1, p.wait_limit, abort_flag)) break;
        uint8_t* st = stage_base + s * S::kStage;
        const int k0 = (kt0 + i) * BK;
        mbar_expect_tx(&full[s], S::kTx);
        for (int mt = 0; mt < MT; ++mt) tma_load_2d(st + mt * 128 * BK * 2, &p.mapA, k0, m0 + mt * 128, &full[s]);
        for (int j = 0; j < BN / 64; ++j)
          tma_load_2d(st + S::kA + j * (BK * 128), &p.mapB[seg], nl + 64 * j, k0, &full[s]);
        ++issued;
      }
      // never leave with copies in flight: wait for the stages still owed
      for (int i = max(0, issued - STAGES); i < issued; ++i) {
        volatile int dummy = 0;
        mbar_wait(&full[i % STAGES], (i / STAGES) & 1, kDrainLimit, &dummy);
      }
      if (*abort_flag) raise(p);
    }
    __syncwarp();   // the warp reaches the CTA barrier below converged
  } else if (warp == 1) {
    // ---- MMA issuer -------------------------------------------------------------
    if (lane == 0) {
      bool ok = true;
      for (int i = 0; i < nk && ok; ++i) {
        const int s = i % STAGES;
        ok = mbar_wait(&full[s], (i / STAGES) & 1, p.wait_limit, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint8_t* a = stage_base + s * S::kStage;
        const uint8_t* b = a + S::kA;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          // B: MN-major, 128-byte swizzle; 64-column blocks 8 KiB apart
          // (leading byte offset), 8-row k groups 1 KiB apart (stride).
          const uint64_t bdesc = smem_desc_sw128(smem_u32(b) + kk * 2048, BK * 128, 1024);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            // A: K-major, 128-byte swizzle, 8-row groups 1 KiB apart; a
            // 16-wide k step moves the start 32 bytes inside the swizzle row.
            const uint64_t adesc = smem_desc_sw128(smem_u32(a + mt * 128 * BK * 2) + kk * 32, 16, 1024);
            mma_f16(tmem_base + mt * BN, adesc, bdesc, kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&empty[s]);
      }
      mma_commit(done);
      if (!ok) raise(p);
    }
    __syncwarp();
  }

  // ---- epilogue: all eight warps ------------------------------------------------------
  {
    const bool ok = mbar_wait(done, 0, p.wait_limit, abort_flag);
    if (!ok) {
      // the MMA thread always commits `done`: wait for its MMAs to finish
      // before the tensor memory they write is freed
      volatile int dummy = 0;
      mbar_wait(done, 0, kDrainLimit, &dummy);
      if (lane == 0) raise(p);
    }
    tc_fence_after();
    // the TMEM loads are warp-collective: the whole warp takes this branch
    if (__all_sync(0xffffffffu, ok && !*abort_flag)) {
      const int q = warp & 3;                        // TMEM lanes 32q .. 32q+31
      const int cb = warp >= 4 ? 0 : BN / 2;         // this warp's half of the columns
      for (int mt = 0; mt < MT; ++mt) {
        const int m = m0 + mt * 128 + q * 32 + lane;
        const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + mt * BN;
        for (int c0 = cb; c0 < cb + BN / 2; c0 += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(trow + c0, r);
          tmem_ld_wait();
          if (m >= p.M) continue;
          const int n = n0 + c0;
          if (p.splits > 1) {
            float4* dst = reinterpret_cast<float4*>(p.partial + (static_cast<size_t>(split) * p.M + m) * p.N + n);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                   __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
          } else {
            float f[32];
#pragma unroll
            for (int v = 0; v < 32; ++v) f[v] = __uint_as_float(r[v]);
            if (p.R) {
              const uint4* rr = reinterpret_cast<const uint4*>(p.R + static_cast<size_t>(m) * p.ldr + n);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const uint4 w = rr[v];
                const __half2* h = reinterpret_cast<const __half2*>(&w);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 x = __half22float2(h[e]);
                  f[8 * v + 2 * e] += x.x;
                  f[8 * v + 2 * e + 1] += x.y;
                }
              }
            }
            if (p.relu) {
#pragma unroll
              for (int v = 0; v < 32; ++v) f[v] = fmaxf(f[v], 0.0f);
            }
            uint4* dst = reinterpret_cast<uint4*>(p.Y + static_cast<size_t>(m) * p.ldy + n);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 w;
              __half2* h = reinterpret_cast<__half2*>(&w);
#pragma unroll
              for (int e = 0; e < 4; ++e) h[e] = __floats2half2_rn(f[8 * v + 2 * e], f[8 * v + 2 * e + 1]);
              dst[v] = w;
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Sum of split-K partials plus the epilogue: Y = relu?(sum_s P[s] + R).
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ part, int splits,
                                                            int M, int N, const __half* __restrict__ R,
                                                            int ldr, int relu, __half* __restrict__ Y,
                                                            int ldy) {
  const int64_t n8 = static_cast<int64_t>(M) * N / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const int64_t e = i * 8;
    const int m = static_cast<int>(e / N), n = static_cast<int>(e % N);
    float f[8];
    {
      const float4 a = *reinterpret_cast<const float4*>(part + e);
      const float4 b = *reinterpret_cast<const float4*>(part + e + 4);
      f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
    for (int s = 1; s < splits; ++s) {
      const float* q = part + static_cast<int64_t>(s) * M * N + e;
      const float4 a = *reinterpret_cast<const float4*>(q);
      const float4 b = *reinterpret_cast<const float4*>(q + 4);
      f[0] += a.x; f[1] += a.y; f[2] += a.z; f[3] += a.w; f[4] += b.x; f[5] += b.y; f[6] += b.z; f[7] += b.w;
    }
    if (R) {
      const uint4 w = *reinterpret_cast<const uint4*>(R + static_cast<int64_t>(m) * ldr + n);
      const __half2* h = reinterpret_cast<const __half2*>(&w);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 x = __half22float2(h[k]);
        f[2 * k] += x.x;
        f[2 * k + 1] += x.y;
      }
    }
    if (relu) {
#pragma unroll
      for (int k = 0; k < 8; ++k) f[k] = fmaxf(f[k], 0.0f);
    }
    uint4 w;
    __half2* h = reinterpret_cast<__half2*>(&w);
#pragma unroll
    for (int k = 0; k < 4; ++k) h[k] = __floats2half2_rn(f[2 * k], f[2 * k + 1]);
    *reinterpret_cast<uint4*>(Y + static_cast<int64_t>(m) * ldy + n) = w;
  }
}

// ---- host side ---------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MT>
fg_status launch(TcParams& p, cudaStream_t st) {
  using S = Smem<MT>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(gemm_tc_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S::kTotal) != cudaSuccess)
      return check_launch("gemm_tc smem attribute");
    attr_set[dev] = true;
  }
  const int grid = p.m_tiles * p.n_tiles * p.splits;
  Trace tr(KC_GEMM_TC, st);
  gemm_tc_kernel<MT><<<grid, kThreads, S::kTotal, st>>>(p);
  return check_launch("gemm_tc_kernel");
}

}  // namespace

bool tc_make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  return make_map(m, dt, base, inner, outer, row_bytes, box_inner, box_outer, sw);
}

// Row tiles per CTA, and the split-K factor of a product (fixed by the shape
// only, so workspace sizes do not depend on the device).
static int tc_mt(int64_t M) { return (M > 128) ? 2 : 1; }

int gemm_tc_splits(int64_t M, int64_t N, int64_t K) {
  const int mt = tc_mt(M);
  const int64_t tiles = ((M + 128 * mt - 1) / (128 * mt)) * (N / BN);
  const int64_t ktiles = K / BK;
  constexpr int64_t kTarget = 148;
  int64_t s = (kTarget + tiles - 1) / tiles;
  if (tiles >= kTarget / 2) s = 1;
  s = s < 1 ? 1 : s;
  const int64_t max_s = ktiles / 4 > 0 ? ktiles / 4 : 1;   // at least 4 k tiles per split
  if (s > max_s) s = max_s;
  if (s > 16) s = 16;
  return static_cast<int>(s);
}

bool gemm_tc_supported(const GemmArgs& a) {
  if (a.dtype != FG_F16 || a.quant) return false;
  if (a.M < 64) return false;
  if (a.K % BK) return false;
  for (int i = 0; i < a.nseg; ++i)
    if (a.seg[i].N % BN || !a.seg[i].dense) return false;
  if ((a.ldx * 2) % 16 || (a.ldy * 2) % 16 || (a.R && (a.ldr * 2) % 16)) return false;
  if (a.M > (1 << 30) || a.N > (1 << 30) || a.K > (1 << 30)) return false;
  return encode_fn() != nullptr;
}

size_t gemm_tc_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const int s = gemm_tc_splits(M, N, K);
  return s > 1 ? static_cast<size_t>(s) * M * N * sizeof(float) : 0;
}

fg_status gemm_tc(const GemmArgs& a, void* ws, size_t ws_bytes, cudaStream_t st) {
  const int mt = tc_mt(a.M);
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.nseg = a.nseg;
  if (!make_map(&p.mapA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.X, a.K, a.M, a.ldx * 2, BK, 128,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return fail(FG_ERR_CUDA, "tensor map for X");
  for (int i = 0; i < a.nseg; ++i) {
    const WSeg& s = a.seg[i];
    p.seg_n0[i] = static_cast<int>(s.n0);
    const bool ok = make_map(&p.mapB[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, s.dense, s.N, a.K, s.N * 2, 64, BK,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return fail(FG_ERR_CUDA, "tensor map for weight segment %d", i);
  }
  p.seg_n0[a.nseg] = static_cast<int>(a.N);
  p.m_tiles = static_cast<int>((a.M + 128 * mt - 1) / (128 * mt));
  p.n_tiles = static_cast<int>(a.N / BN);
  {
    // no split may be empty: derive the count back from the per-split length
    const int ktiles = static_cast<int>(a.K / BK);
    const int want = gemm_tc_splits(a.M, a.N, a.K);
    p.ktiles_per_split = (ktiles + want - 1) / want;
    p.splits = (ktiles + p.ktiles_per_split - 1) / p.ktiles_per_split;
  }
  p.group_n = 8;
  p.Y = static_cast<__half*>(a.Y);
  p.ldy = static_cast<int>(a.ldy);
  p.R = static_cast<const __half*>(a.R);
  p.ldr = static_cast<int>(a.ldr);
  p.relu = a.relu;
  p.err = device_error_word();
  if (!p.err) return fail(FG_ERR_CUDA, "device error word");
  p.wait_limit = wait_limit();
  if (p.splits > 1) {
    const size_t need = static_cast<size_t>(p.splits) * a.M * a.N * sizeof(float);
    if (!ws || ws_bytes < need) return fail(FG_ERR_WORKSPACE, "split-K partials need %zu bytes", need);
    p.partial = static_cast<float*>(ws);
  }
  const fg_status s = mt == 1 ? launch<1>(p, st) : launch<2>(p, st);
  if (s != FG_OK || p.splits == 1) return s;
  const int64_t n8 = a.M * a.N / 8;
  int grid = static_cast<int>((n8 + 255) / 256);
  if (grid > num_sms() * 8) grid = num_sms() * 8;
  Trace tr(KC_GEMM_REDUCE, st);
  splitk_reduce_kernel<<<grid, 256, 0, st>>>(p.partial, p.splits, p.M, p.N, p.R, p.ldr, p.relu, p.Y, p.ldy);
  return check_launch("splitk_reduce_kernel");
}

}  // namespace fg
