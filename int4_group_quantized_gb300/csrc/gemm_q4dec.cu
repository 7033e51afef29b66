// Decode products on 4-bit weights: Y = epilogue(X . W) for a block of
// M <= 256 sequences (FlexGen notes, "4. 卸载策略": zig-zag block, one read
// of a layer's weights for the whole block; "5. 近似方法": 4-bit groups of 64
// along the output channel, converted back to FP16 before compute).
//
// Here the weights are the M = 128 operand of tcgen05.mma and the block of
// activations is the N operand (Y^T = W^T X^T), so nothing is padded:
//   * A = 128 output channels x 64 k, fp16, MN-major (channels contiguous,
//     128-byte swizzle), written by eight dequantization warps from the
//     4-bit codes and (min, scale) pairs that TMA brings in;
//   * B = X tile [BT rows][64 k], K-major, 128-byte swizzle, by TMA (rows
//     past M zero-filled);
//   * the accumulator is 128 TMEM lanes (channels) x BT columns (sequences).
// Each weight byte crosses HBM once per step; the kernel is HBM-bound, so the
// CTA is small enough for two per SM and splits K when the output has too
// few 128-channel tiles to fill the GPU.  The K splits of a tile form one
// thread-block cluster and sum their partials over distributed shared memory
// in the same launch.
//
// Warp roles (384 threads): warp 0 issues TMA, warp 1 owns TMEM and issues
// the MMAs, warps 4..11 dequantize, warps 4..7 drain TMEM.  Every wait is
// bounded and raises the device error word on timeout.
#include <cudaTypedefs.h>
#include <string.h>

#include <cooperative_groups.h>

#include "fg_internal.cuh"
#include "q4_dev.cuh"
#include "tc_ptx.cuh"

namespace fg {

// defined in gemm_tc.cu
bool tc_make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

namespace {

using namespace tc;
using namespace q4;
namespace cg = cooperative_groups;

constexpr int BK = 64;
constexpr int BNC = 128;               // output channels per CTA (the MMA's M)
constexpr int kThreads = 384;
constexpr int kDqWarp0 = 4;            // warps 4..11
constexpr int kDqThreads = kThreads - 32 * kDqWarp0;
constexpr int kEpiWarp0 = 4;           // warps 4..7: TMEM lanes 0..127
constexpr uint32_t kWaitLimit = 1u << 24;

struct DecParams {
  CUtensorMap mapX;
  CUtensorMap mapC[3], mapMin[3], mapScale[3];
  int seg_n0[4];
  int nseg;
  int M, N, K;
  int n_tiles, splits, ktiles_per_split;
  __half* Y;
  int ldy;
  const __half* R;
  int ldr;
  int relu;
  unsigned int* err;
};

template <int BT>
struct DecSmem {
  static constexpr int kX = BT * BK * 2;
  static constexpr int kCodes = BK * BNC / 2;
  static constexpr int kMeta = BK * 4 * 4;           // 4 floats (256 channels) per row, 16-byte boxes
  static constexpr int kTx = kX + kCodes + 2 * kMeta;
  static constexpr int kStage = (kTx + 1023) / 1024 * 1024;
  static constexpr int kW = BK * BNC * 2;            // one dequantized weight tile
  static constexpr int kNW = BT <= 128 ? 3 : 3;
  static constexpr int kBudget = BT <= 128 ? 104 * 1024 : 200 * 1024;   // two CTAs per SM up to BT = 128
  static constexpr int kStages = (kBudget - kNW * kW) / kStage > 6 ? 6 : (kBudget - kNW * kW) / kStage;
  static constexpr int kTotal = 1024 + kStages * kStage + kNW * kW + 256;
  static_assert(kStages >= 2, "pipeline needs two stages");
};

template <int BT>
__global__ void __launch_bounds__(kThreads, 1) gemm_q4_decode_kernel(const __grid_constant__ DecParams p) {
  using S = DecSmem<BT>;
  constexpr int STAGES = S::kStages;
  constexpr int NW = S::kNW;
  constexpr uint32_t kTmemCols = BT < 32 ? 32 : BT;
  constexpr uint32_t kIdesc = idesc_f16(128, BT, 1, 0);   // A MN-major (weights), B K-major (X)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  uint8_t* wbuf = smem + STAGES * S::kStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(wbuf + NW * S::kW);
  uint64_t* empty = full + STAGES;
  uint64_t* wfull = empty + STAGES;
  uint64_t* wempty = wfull + NW;
  uint64_t* done = wempty + NW;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x % p.splits;
  const int nt = blockIdx.x / p.splits;
  const int n0 = nt * BNC;
  int seg = 0;
  while (seg + 1 < p.nseg && n0 >= p.seg_n0[seg + 1]) ++seg;
  const int nl = n0 - p.seg_n0[seg];
  const int kt0 = split * p.ktiles_per_split;
  const int kt1 = min(kt0 + p.ktiles_per_split, p.K / BK);
  const int nk = kt1 - kt0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1 + kDqThreads / 32);   // the MMA commit + one arrival per dequant warp
    }
    for (int i = 0; i < NW; ++i) {
      mbar_init(&wfull[i], kDqThreads / 32);
      mbar_init(&wempty[i], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.mapX);
    tma_prefetch_desc(&p.mapC[seg]);
    tma_prefetch_desc(&p.mapMin[seg]);
    tma_prefetch_desc(&p.mapScale[seg]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(&empty[s], ((i / STAGES) & 1) ^ 1, kWaitLimit, abort_flag)) break;
        uint8_t* st = stage_base + s * S::kStage;
        const int k0 = (kt0 + i) * BK;
        mbar_expect_tx(&full[s], S::kTx);
        tma_load_2d(st, &p.mapX, k0, 0, &full[s]);
        tma_load_2d(st + S::kX, &p.mapC[seg], nl / 2, k0, &full[s]);
        tma_load_2d(st + S::kX + S::kCodes, &p.mapMin[seg], (nl / 256) * 4, k0, &full[s]);
        tma_load_2d(st + S::kX + S::kCodes + S::kMeta, &p.mapScale[seg], (nl / 256) * 4, k0, &full[s]);
        ++issued;
      }
      for (int i = max(0, issued - STAGES); i < issued; ++i) {
        volatile int dummy = 0;
        mbar_wait(&full[i % STAGES], (i / STAGES) & 1, kWaitLimit, &dummy);
      }
      if (*abort_flag) atomicOr(p.err, DEV_ERR_WAIT_TIMEOUT);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = true;
      for (int i = 0; i < nk && ok; ++i) {
        const int s = i % STAGES;
        const int j = i % NW;
        ok = mbar_wait(&full[s], (i / STAGES) & 1, kWaitLimit, abort_flag) &&
             mbar_wait(&wfull[j], (i / NW) & 1, kWaitLimit, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t xa = smem_u32(stage_base + s * S::kStage);
        const uint32_t wa = smem_u32(wbuf + j * S::kW);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          // A (weights): MN-major, 64-channel blocks 8 KiB apart, 8-row k groups 1 KiB apart
          const uint64_t adesc = smem_desc_sw128(wa + kk * 2048, BK * 128, 1024);
          // B (X): K-major, 8-row groups 1 KiB apart; +32 bytes per 16-wide k step
          const uint64_t bdesc = smem_desc_sw128(xa + kk * 32, 16, 1024);
          mma_f16(tmem_base, adesc, bdesc, kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&empty[s]);
        mma_commit(&wempty[j]);
      }
      mma_commit(done);
      if (!ok) atomicOr(p.err, DEV_ERR_WAIT_TIMEOUT);
    }
  } else if (warp >= kDqWarp0) {
    const int t = threadIdx.x - 32 * kDqWarp0;
    const int g0 = (nl & 255) >> 6;
    bool ok = true;
    for (int i = 0; i < nk && ok; ++i) {
      const int s = i % STAGES;
      const int j = i % NW;
      ok = mbar_wait(&full[s], (i / STAGES) & 1, kWaitLimit, abort_flag) &&
           mbar_wait(&wempty[j], ((i / NW) & 1) ^ 1, kWaitLimit, abort_flag);
      if (!ok) break;
      const uint8_t* st = stage_base + s * S::kStage;
      const uint2* codes = reinterpret_cast<const uint2*>(st + S::kX);
      const float* mins = reinterpret_cast<const float*>(st + S::kX + S::kCodes);
      const float* scales = mins + BK * 4;
      uint8_t* w = wbuf + j * S::kW;
      constexpr int kUnits = BK * BNC / 16;
      static_assert(kUnits % kDqThreads == 0, "units split evenly");
#pragma unroll
      for (int it = 0; it < kUnits / kDqThreads; ++it) {
        const int u = t + it * kDqThreads;
        const int k = u / (BNC / 16);
        const int n = (u % (BNC / 16)) * 16;
        const int gi = k * 4 + g0 + n / 64;
        const uint32_t s2 = bcast_h2(scales[gi]), m2 = bcast_h2(mins[gi]);
        const uint2 c = codes[k * (BNC / 16) + n / 16];
        const uint4 v0 = dequant8(c.x, s2, m2);
        const uint4 v1 = dequant8(c.y, s2, m2);
        const int chunk = (n & 63) >> 3;
        uint8_t* row = w + (n >> 6) * (BK * 128) + k * 128;
        *reinterpret_cast<uint4*>(row + ((chunk ^ (k & 7)) << 4)) = v0;
        *reinterpret_cast<uint4*>(row + (((chunk + 1) ^ (k & 7)) << 4)) = v1;
      }
      // each thread orders its own stores before the tensor core reads them;
      // the warp then signals once
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&wfull[j]);
        mbar_arrive(&empty[s]);
      }
    }
  }

  // ---- epilogue: TMEM lane = channel, column = sequence ---------------------------
  // With one split the accumulator goes straight to Y.  With several, the
  // splits of a tile form one thread-block cluster: each CTA parks its fp32
  // partial in its own shared memory (the drained pipeline buffers), and
  // after a cluster barrier CTA r sums rows [r*M/splits, ...) of all the
  // partials over distributed shared memory and writes them.
  const bool direct = p.splits == 1;
  float* part = reinterpret_cast<float*>(stage_base);     // [BT][128] fp32
  if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    const int q = warp - kEpiWarp0;
    const int r = 32 * q + lane;                           // A row = TMEM lane
    const int ch = n0 + (r & ~7) + perm8(r & 7);           // output channel of this lane
    bool ok = mbar_wait(done, 0, kWaitLimit, abort_flag);
    tc_fence_after();
    ok = ok && !*abort_flag;
#pragma unroll 1
    for (int c0 = 0; c0 < BT; c0 += 32) {
      uint32_t v[32];
      tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + c0, v);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int m = c0 + e;
        const float f = ok ? __uint_as_float(v[e]) : 0.0f;
        if (direct) {
          if (m < p.M && ok) {
            float y = f;
            if (p.R) y += __half2float(p.R[static_cast<size_t>(m) * p.ldr + ch]);
            if (p.relu) y = fmaxf(y, 0.0f);
            p.Y[static_cast<size_t>(m) * p.ldy + ch] = __float2half_rn(y);
          }
        } else {
          part[m * BNC + r] = f;
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
  if (!direct) {
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();   // every split's partial is in its CTA's shared memory
    const int rk = static_cast<int>(cl.block_rank());
    const int rows = (p.M + p.splits - 1) / p.splits;
    const int mlo = rk * rows, mhi = min(p.M, mlo + rows);
    for (int e = threadIdx.x; e < (mhi - mlo) * BNC; e += kThreads) {
      const int m = mlo + e / BNC, r = e % BNC;
      float f = 0.0f;
      for (int s = 0; s < p.splits; ++s) f += cl.map_shared_rank(part, s)[m * BNC + r];
      const int ch = n0 + (r & ~7) + perm8(r & 7);
      if (p.R) f += __half2float(p.R[static_cast<size_t>(m) * p.ldr + ch]);
      if (p.relu) f = fmaxf(f, 0.0f);
      p.Y[static_cast<size_t>(m) * p.ldy + ch] = __float2half_rn(f);
    }
    cl.sync();   // no CTA leaves while a peer may still read its partial
  }
}

template <int BT>
fg_status launch_dec(DecParams& p, cudaStream_t st) {
  using S = DecSmem<BT>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(gemm_q4_decode_kernel<BT>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kTotal) !=
        cudaSuccess)
      return check_launch("gemm_q4_decode smem attribute");
    attr_set[dev] = true;
  }
  Trace tr(KC_GEMM_TC, st);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.n_tiles * p.splits));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = S::kTotal;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;   // the K splits of a tile share a cluster
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gemm_q4_decode_kernel<BT>, p) != cudaSuccess)
    return check_launch("gemm_q4_decode_kernel (cluster launch)");
  return check_launch("gemm_q4_decode_kernel");
}

int bt_for(int64_t M) { return M <= 64 ? 64 : (M <= 128 ? 128 : 256); }

}  // namespace

// Split count for a decode product: K is cut so that the CTAs fill the
// GPU's slots (two per SM up to 128 sequences) with the fewest waves of
// per-CTA work; depends on the shape only.
int gemm_q4dec_splits(int64_t M, int64_t N, int64_t K) {
  const int64_t tiles = N / BNC, ktiles = K / BK;
  const int64_t slots = (M <= 128 ? 2 : 1) * static_cast<int64_t>(num_sms());
  int64_t best = 1;
  double best_cost = 1e30;
  for (int64_t s = 1; s <= 8 && s <= ktiles / 2; ++s) {   // a cluster holds at most 8 CTAs
    const int64_t waves = (tiles * s + slots - 1) / slots;
    const double cost = static_cast<double>(waves) * ((ktiles + s - 1) / s) + 0.5 * s;
    if (cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return static_cast<int>(best);
}

bool gemm_q4dec_supported(const GemmArgs& a) {
  if (a.dtype != FG_F16 || !a.quant || a.M < 1 || a.M > 256 || a.K % BK) return false;
  for (int i = 0; i < a.nseg; ++i) {
    if (a.seg[i].N % BNC) return false;
    if (((a.seg[i].N / 64) * 4) % 16) return false;
    if (!aligned(a.seg[i].codes, 16) || !aligned(a.seg[i].mins, 16) || !aligned(a.seg[i].scales, 16)) return false;
  }
  if ((a.ldx * 2) % 16) return false;
  return true;
}

fg_status gemm_q4dec(const GemmArgs& a, cudaStream_t st) {
  DecParams p;
  memset(&p, 0, sizeof(p));
  const int bt = bt_for(a.M);
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.nseg = a.nseg;
  if (!tc_make_map(&p.mapX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.X, a.K, a.M, a.ldx * 2, BK, bt,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return fail(FG_ERR_CUDA, "tensor map for X");
  for (int i = 0; i < a.nseg; ++i) {
    const WSeg& s = a.seg[i];
    p.seg_n0[i] = static_cast<int>(s.n0);
    const bool ok =
        tc_make_map(&p.mapC[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, s.codes, s.N / 2, a.K, s.N / 2, BNC / 2, BK,
                    CU_TENSOR_MAP_SWIZZLE_NONE) &&
        tc_make_map(&p.mapMin[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, s.mins, s.N / 64, a.K, (s.N / 64) * 4, 4, BK,
                    CU_TENSOR_MAP_SWIZZLE_NONE) &&
        tc_make_map(&p.mapScale[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, s.scales, s.N / 64, a.K, (s.N / 64) * 4, 4,
                    BK, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) return fail(FG_ERR_CUDA, "tensor map for weight segment %d", i);
  }
  p.seg_n0[a.nseg] = static_cast<int>(a.N);
  p.n_tiles = static_cast<int>(a.N / BNC);
  {
    const int ktiles = static_cast<int>(a.K / BK);
    const int want = gemm_q4dec_splits(a.M, a.N, a.K);
    p.ktiles_per_split = (ktiles + want - 1) / want;
    p.splits = (ktiles + p.ktiles_per_split - 1) / p.ktiles_per_split;
  }
  p.Y = static_cast<__half*>(a.Y);
  p.ldy = static_cast<int>(a.ldy);
  p.R = static_cast<const __half*>(a.R);
  p.ldr = static_cast<int>(a.ldr);
  p.relu = a.relu;
  p.err = device_error_word();
  if (!p.err) return fail(FG_ERR_CUDA, "device error word");
  switch (bt) {
    case 64: return launch_dec<64>(p, st);
    case 128: return launch_dec<128>(p, st);
    default: return launch_dec<256>(p, st);
  }
}

}  // namespace fg
