// Decode products on 4-bit weights with the weights in tensor memory
// (FlexGen notes, "4. 卸载策略": zig-zag block, one read of a layer's weights
// serves every sequence of the block; "5. 近似方法": 4-bit groups of 64 along
// the output channel, converted back to FP16 before compute).
//
// Y^T = W^T X^T on tcgen05.mma kind::f16 with A taken from TMEM.  A CTA
// owns RB row blocks of 128 output channels (RB = 2: one CTA per SM with all
// 512 TMEM columns; RB = 1: two CTAs per SM):
//   * A = 128 channels x 64 k per row block.  Dequantization warps turn the
//     packed codes and (scale, min) pairs of the decode copy (fg_pack_weight)
//     into fp16 weights in registers and store them with tcgen05.st: with the
//     stored fp32 pairs each weight is fp16(fmaf(q, scale, min)), exactly the
//     value the format's dequantization gives; with the opt-in fp16 pairs it
//     is fp16(q * scale' + min') in one fp16 FMA.  TMEM lane =
//     channel, column = two consecutive k.  A warp reaches only its own
//     32-lane quarter of TMEM (warp % 4); two sets of 4*RB warps convert
//     the two k tiles of a chunk side by side.
//   * B = X tile [BT rows][64 k], K-major, 128-byte swizzle, by TMA, shared
//     by the RB row blocks: the activations cross L2 once per 128*RB
//     channels, which is what bounds this kernel at small RB.
//   * D = RB accumulators of 128 lanes (channels) x BT columns (sequences).
// Shared memory carries only what HBM delivers (codes, pairs) and X; the fp16
// weights never touch it.
//
// K is split when there are too few channel tiles to fill the GPU.  The
// splits of a channel tile form one thread-block cluster: each stages its
// fp32 partial [M][128] in its own shared memory, then the cluster's CTAs
// share the rows of the output, each summing every split's partial of its
// rows over distributed shared memory in split (rank) order and applying the
// epilogue.  No partial goes through global memory and no second kernel
// runs.
//
// The kernel is launched with programmatic stream serialization: the weight
// tiles of the first stages are requested and converted before
// griddepcontrol.wait, so they stream while the previous kernel finishes; X,
// the residual, the workspace and Y are touched only after it.
//
// Warp roles (128 + 256*RB threads): warp 0 issues the weight copies, warp 2
// the X copies, warp 1 owns TMEM and issues the MMAs, warp 3 (the sync warp)
// waits on the copies' mbarriers for the converting warps, warps 4..
// dequantize, and the first 4*RB of them drain TMEM.  Every mbarrier wait is
// bounded and raises the device error word on timeout; each named barrier is
// taken the same number of times by all of its warps.
#include <cudaTypedefs.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#include "fg_internal.cuh"
#include "q4_convert.cuh"
#include "q4_dev.cuh"
#include "tc_ptx.cuh"

namespace fg {

// defined in gemm_tc.cu
bool tc_make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

namespace {

using namespace tc;
using namespace q4;

constexpr int BK = 64;
constexpr int BNC = 128;               // channels per row block (the MMA's M)
constexpr int kDqWarp0 = 4;            // dequantization warps start here
constexpr int kMaxSplits = 8;          // K splits of a decode product: a portable cluster
// The copy producers run stages ahead and usually find their ring full; they
// poll with this pause so that they leave the issue slots to the converters.
constexpr uint32_t kProducerSleepNs = 100;

// ---- packing -------------------------------------------------------------------
// The decode copy is one block per (128-channel tile nt, 64-k tile kt), blocks
// in order nt-major, so a CTA streams one contiguous run of HBM and fetches a
// stage with one bulk copy.  Inside a block the data sit where the thread
// that converts them reads them, for the 16x128b TMEM store shape (warp
// quarter q writes TMEM lanes 32q..32q+31 with two stores of 16 lanes; thread
// t of the warp holds lanes t/4, t/4+8, t/4+16, t/4+24 and the 32-bit columns
// c = t%4, t%4+4, ..., i.e. the k pairs j = 4i + t%4, i = 0..7):
//   bytes 0..4095: codes, [q][g2][t] 16-byte units (q = 0..3, g2 = 0..1,
//     t = 0..31): word w of unit (q, g2, t) is channel 32q + t/4 + 8w, k pairs
//     j = 16*g2 + 4e + t%4 for e = 0..3, nibble slot e (from the low end)
//     holding k = 2j and slot e+4 holding k = 2j+1.  A warp's 128-bit loads
//     are 512 contiguous bytes each.
//   then the (scale, min) pairs of the tile's two 64-channel groups gl:
//   * FG_PACK_EXACT (1024 bytes): the 16-byte unit gl*512 + j*16 holds fp32
//     (scale[2j], scale[2j+1], min[2j], min[2j+1]) as stored; a warp's load
//     of unit j = 4i + t%4 touches 4 distinct units (64 contiguous bytes);
//   * FG_PACK_F16META (512 bytes): [gl][u][c4] 16-byte units, u = 0..3,
//     c4 = 0..3: fp16x2 (scale[2j], scale[2j+1]), fp16x2 (min[2j],
//     min[2j+1]) for j = 8u + c4, then the same for j = 8u + 4 + c4.
constexpr int kTileCodes = BNC * BK / 2;             // 4096

__host__ __device__ constexpr int tile_bytes(int fmt) {
  return kTileCodes + (fmt == FG_PACK_EXACT ? 2 * (BK / 2) * 16 : 2 * (BK / 2) * 8);   // 5120 or 4608
}

__global__ void pack_codes_kernel(const uint8_t* __restrict__ codes, int64_t K, int64_t N, int tb,
                                  uint8_t* __restrict__ packed) {
  const int64_t words = N * (K / 8), KT = K / BK;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < words;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = i % N, rest = i / N;   // threads along n: coalesced reads of a code row
    const int c4 = static_cast<int>(rest % 4), g2 = static_cast<int>((rest / 4) % 2);
    const int64_t kt = rest / 8;
    const int r = static_cast<int>(n % BNC);
    const int q = r / 32, w = (r % 32) / 8, t = ((r % 8) << 2) | c4;
    uint32_t out = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t k = kt * BK + 2 * (16 * g2 + 4 * e + c4);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t byte = codes[(k + h) * (N / 2) + n / 2];
        const uint32_t c = (n & 1) ? (byte >> 4) : (byte & 15u);
        out |= c << (4 * (e + 4 * h));
      }
    }
    uint8_t* tile = packed + ((n / BNC) * KT + kt) * tb;
    *reinterpret_cast<uint32_t*>(tile + q * 1024 + g2 * 512 + t * 16 + w * 4) = out;
  }
}

// FG_PACK_F16META pairs: (scale, min) rounded to fp16, nearest even.
__global__ void pack_pairs_f16_kernel(const float* __restrict__ mins, const float* __restrict__ scales, int64_t K,
                                      int64_t N, uint8_t* __restrict__ packed) {
  constexpr int tb = tile_bytes(FG_PACK_F16META);
  const int64_t G = N / 64, total = G * (K / 2), KT = K / BK;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t g = i % G, jj = i / G;     // jj = global k pair; threads along g: coalesced reads
    const __half2 s2 = __floats2half2_rn(scales[(2 * jj) * G + g], scales[(2 * jj + 1) * G + g]);
    const __half2 m2 = __floats2half2_rn(mins[(2 * jj) * G + g], mins[(2 * jj + 1) * G + g]);
    const int64_t kt = jj / (BK / 2);
    const int j = static_cast<int>(jj % (BK / 2));
    const int u = j / 8, hi = (j / 4) % 2, c4 = j % 4;
    uint8_t* tile = packed + ((g / 2) * KT + kt) * tb;
    *reinterpret_cast<uint2*>(tile + kTileCodes + (g % 2) * 256 + (u * 4 + c4) * 16 + hi * 8) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&s2), *reinterpret_cast<const uint32_t*>(&m2));
  }
}

// FG_PACK_EXACT pairs: the stored fp32 values, regrouped per k pair.
__global__ void pack_pairs_f32_kernel(const float* __restrict__ mins, const float* __restrict__ scales, int64_t K,
                                      int64_t N, uint8_t* __restrict__ packed) {
  constexpr int tb = tile_bytes(FG_PACK_EXACT);
  const int64_t G = N / 64, total = G * (K / 2), KT = K / BK;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t g = i % G, jj = i / G;
    const float4 v = make_float4(scales[(2 * jj) * G + g], scales[(2 * jj + 1) * G + g], mins[(2 * jj) * G + g],
                                 mins[(2 * jj + 1) * G + g]);
    const int64_t kt = jj / (BK / 2);
    const int j = static_cast<int>(jj % (BK / 2));
    uint8_t* tile = packed + ((g / 2) * KT + kt) * tb;
    *reinterpret_cast<float4*>(tile + kTileCodes + (g % 2) * 512 + j * 16) = v;
  }
}

struct TsParams {
  CUtensorMap mapX;
  const uint8_t* wp[3];     // decode copy of each segment
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
  uint32_t wait_limit;      // polls of a bounded wait (fg_set_wait_limit)
};

constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int cmax(int a, int b) { return a > b ? a : b; }

// The main loop runs in lockstep chunks of kT k tiles.  The dequantization
// warps (kT sets of 4*RB, one k tile of the chunk each) convert chunk c into
// TMEM buffer c % kBufs and meet the MMA warp at one hardware named barrier;
// the MMA warp then issues chunk c's MMAs while the dequantization warps
// convert chunk c+1.  One barrier per chunk replaces a handoff per k tile:
// on this GPU every synchronisation the issuing thread takes (an mbarrier
// wait, an acquire load) costs a few hundred cycles, about the MMA time of a
// whole k tile at N = 64.  Every warp that takes the named barrier runs the
// same number of chunks and leaves the loop only at its end, so the barrier
// always completes; a failed (bounded) wait skips the work, not the barrier.
//
// The dequantization warps touch no mbarrier: a sync warp takes every wait
// on their behalf before each chunk barrier (the chunk's X tiles, the next
// TMEM buffer free, the weights two chunks ahead) and releases the weight
// stages they have converted after it.  They are software-pipelined by one
// chunk: chunk c+1 is loaded and converted while chunk c's stores complete.
//
// Rings around it, each released by the stage that last needs it: weights
// (a chunk's packed blocks, one bulk copy per row block; released once every
// dequantization warp holds its codes in registers), X (a chunk's tiles) and
// the TMEM buffers (both released by the commit of the MMAs that read them).
template <int BT, int RB, int FMT>
struct TsCfg {
  static constexpr int kTileBytes = tile_bytes(FMT);
  static constexpr int kT = 2;                        // k tiles per chunk
  static constexpr int kGroupWarps = 4 * RB;          // warps converting one k tile (all row blocks)
  static constexpr int kDqWarps = kT * kGroupWarps;
  static constexpr int kThreads = 128 + kDqWarps * 32;   // warps 0..3, then the dequantization warps
  static constexpr int kBarThreads = 64 + kDqWarps * 32;   // MMA warp, sync warp, dequantization warps
  static constexpr int kStartThreads = 32 + kDqWarps * 32; // sync warp, dequantization warps
  static constexpr int kX = BT * BK * 2;              // X tile, K-major, 128-byte swizzle
  static constexpr int kXStage = kT * kX;
  static constexpr int kWStage = kT * RB * kTileBytes;   // a chunk's packed blocks, [rb][t]
  static constexpr int kAcc = BT < 32 ? 32 : BT;      // accumulator columns per row block
  static constexpr int kBufCols = 32 * RB * kT;       // TMEM columns of one A buffer
  static constexpr uint32_t kTmemCols = (RB == 1 && BT <= 128) ? 256 : 512;
  static constexpr int kMinBlocks = kTmemCols == 256 ? 2 : 1;
  static constexpr int kBudget = kMinBlocks == 2 ? 104 * 1024 : 204 * 1024;
  // TMEM A buffers, and X stages (no more than the buffers: every parity
  // wait on a buffer's commit barrier then sees its phase before the next)
  static constexpr int kBufs = cmin(4, (static_cast<int>(kTmemCols) - RB * kAcc) / kBufCols);
  static constexpr int kXStages = cmax(2, cmin(kBufs, (kBudget * 5 / 8) / kXStage));
  static constexpr int kWStages = cmin(8, (kBudget - kXStages * kXStage) / kWStage);
  static constexpr int kXBytes = kXStages * kXStage;
  static constexpr int kWBytes = kWStages * kWStage;
  static constexpr int kBarBytes = (kXStages + 2 * kWStages + kBufs + 1) * 8 + 16;   // + done, TMEM slot, flag
  static constexpr int kTotal = 1024 + kXBytes + kWBytes + kBarBytes;
  static_assert(kBufs >= 2 && kWStages >= 2, "pipeline needs two stages");
  static_assert(kXStages <= kBufs, "X stages are freed by buffer commits");
  static_assert(kX % 1024 == 0, "X tiles stay 1024-byte aligned");
  static_assert(kXBytes + kWBytes >= BT * RB * BNC * 4, "a split partial is staged in the drained rings");
};

constexpr uint32_t kChunkBarrier = 1;   // named barrier ids (0 is __syncthreads)
constexpr uint32_t kStartBarrier = 2;
constexpr int kSyncWarp = 3;

template <int BT, int RB, int FMT>
__global__ void __launch_bounds__(TsCfg<BT, RB, FMT>::kThreads, TsCfg<BT, RB, FMT>::kMinBlocks)
    gemm_q4ts_kernel(const __grid_constant__ TsParams p) {
  using C = TsCfg<BT, RB, FMT>;
  constexpr int kTileBytes = C::kTileBytes;
  constexpr int KT = C::kT, NB = C::kBufs, SX = C::kXStages, SW = C::kWStages;
  constexpr uint32_t kIdesc = idesc_f16(128, BT, 0, 0);   // A (TMEM) and B (X) K-major
  constexpr uint32_t kACol = RB * C::kAcc;                // TMEM A buffers follow the accumulators

  extern __shared__ uint8_t smem_raw[];
  uint8_t* xring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wring = xring + C::kXBytes;
  // xfull[x]: X stage x has landed (chunk c uses stage c % SX); it is
  // requested once the MMAs of chunk c - SX, the last to read it, completed
  uint64_t* xfull = reinterpret_cast<uint64_t*>(wring + C::kWBytes);
  uint64_t* wfull = xfull + SX;
  uint64_t* wempty = wfull + SW;     // one arrival per dequantization warp
  uint64_t* bufdone = wempty + SW;   // TMEM A buffer read by its MMAs
  uint64_t* done = bufdone + NB;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x % p.splits;
  const int nt = blockIdx.x / p.splits;
  const int n0 = nt * BNC * RB;
  int seg = 0;
  while (seg + 1 < p.nseg && n0 >= p.seg_n0[seg + 1]) ++seg;
  const int nl = n0 - p.seg_n0[seg];
  const int kt0 = split * p.ktiles_per_split;
  const int kt1 = min(kt0 + p.ktiles_per_split, p.K / BK);
  const int nk = kt1 - kt0;
  const int nch = (nk + KT - 1) / KT;

  griddep_launch();   // a dependent grid waits for this one before it reads Y

  if (threadIdx.x == 0) {
    for (int i = 0; i < SX; ++i) mbar_init(&xfull[i], 1);
    for (int i = 0; i < SW; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], 1);        // the sync warp, once every warp has converted the stage
    }
    for (int i = 0; i < NB; ++i) mbar_init(&bufdone[i], 1);   // the MMA commit
    mbar_init(done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  if (warp == 2 && lane == 0) tma_prefetch_desc(&p.mapX);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // weights: independent of the previous kernel, so they stream from the start;
      // the k tiles of a 128-channel block are one contiguous run of packed blocks
      const size_t run = static_cast<size_t>(p.K / BK) * kTileBytes;
      const uint8_t* wsrc = p.wp[seg] + static_cast<size_t>(nl / BNC) * run + static_cast<size_t>(kt0) * kTileBytes;
      int issued = 0;
      for (int c = 0; c < nch; ++c) {
        const int s = c % SW;
        const uint32_t bytes = static_cast<uint32_t>(min(KT, nk - KT * c) * kTileBytes);
        if (!mbar_wait_sleep(&wempty[s], ((c / SW) & 1) ^ 1, p.wait_limit, abort_flag, kProducerSleepNs)) break;
        mbar_expect_tx(&wfull[s], bytes * RB);
#pragma unroll
        for (int rb = 0; rb < RB; ++rb)
          bulk_load(wring + s * C::kWStage + rb * KT * kTileBytes,
                    wsrc + rb * run + static_cast<size_t>(KT * c) * kTileBytes, bytes, &wfull[s]);
        ++issued;
      }
      for (int c = max(0, issued - SW); c < issued; ++c) {   // nothing in flight at exit
        volatile int dummy = 0;
        mbar_wait(&wfull[c % SW], (c / SW) & 1, kDrainLimit, &dummy);
      }
      if (*abort_flag) atomicOr(p.err, DEV_ERR_WAIT_TIMEOUT);
    }
    __syncwarp();   // the warp reaches the CTA barriers below converged
  } else if (warp == 2) {
    if (lane == 0) {
      griddep_wait();   // X comes from the previous kernel
      int issued = 0;
      for (int c = 0; c < nch; ++c) {
        const int s = c % SX, n = min(KT, nk - KT * c);
        // the MMAs of chunk c - SX, the last to read stage s, have completed
        if (c >= SX && !mbar_wait_sleep(&bufdone[(c - SX) % NB], ((c - SX) / NB) & 1, p.wait_limit, abort_flag,
                                        kProducerSleepNs))
          break;
        mbar_expect_tx(&xfull[s], n * C::kX);
        for (int t = 0; t < n; ++t)
          tma_load_2d(xring + s * C::kXStage + t * C::kX, &p.mapX, (kt0 + KT * c + t) * BK, 0, &xfull[s]);
        ++issued;
      }
      for (int c = max(0, issued - SX); c < issued; ++c) {
        volatile int dummy = 0;
        mbar_wait(&xfull[c % SX], (c / SX) & 1, kDrainLimit, &dummy);
      }
      if (*abort_flag) atomicOr(p.err, DEV_ERR_WAIT_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // every lane takes the barrier; lane 0 issues
    for (int c = 0; c < nch; ++c) {
      const int n = min(KT, nk - KT * c);
      named_bar_sync(kChunkBarrier, C::kBarThreads);   // chunk c is in TMEM and its X tiles have landed
      if (lane == 0) {
        tc_fence_after();
        const int b = c % NB;
        if (!*abort_flag) {
          for (int t = 0; t < n; ++t) {
            const uint32_t xa = smem_u32(xring + (c % SX) * C::kXStage + t * C::kX);
#pragma unroll
            for (int rb = 0; rb < RB; ++rb) {
              const uint32_t ta = tmem_base + kACol + b * C::kBufCols + 32u * (t * RB + rb);
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                // B (X): K-major, 8-row groups 1 KiB apart; +32 bytes per 16-wide k step
                const uint64_t bdesc = smem_desc_sw128(xa + kk * 32, 16, 1024);
                mma_f16_ts(tmem_base + rb * C::kAcc, ta + 8u * kk, bdesc, kIdesc, (c > 0 || t > 0 || kk > 0) ? 1u : 0u);
              }
            }
          }
        }
        mma_commit(&bufdone[b]);   // frees X stage b and TMEM buffer b
      }
      __syncwarp();
    }
    if (lane == 0) {
      mma_commit(done);
      if (*abort_flag) atomicOr(p.err, DEV_ERR_WAIT_TIMEOUT);
    }
  } else if (warp == kSyncWarp) {
    // Waits, on behalf of the warps that take the chunk barrier, for what
    // comes after it, so that the dequantization warps touch no mbarrier:
    // before chunk barrier c, chunk c's X tiles (for the MMA warp), TMEM
    // buffer (c+1) % NB free (the MMAs of chunk c+1-NB done) and the weights
    // of chunk c+2 (for the converting warps); after it, releases the weight
    // stages that have been converted by then.
    bool ok = nch > 0 && mbar_wait(&wfull[0], 0, p.wait_limit, abort_flag) &&
              (nch < 2 || mbar_wait(&wfull[1 % SW], (1 / SW) & 1, p.wait_limit, abort_flag));
    named_bar_sync(kStartBarrier, C::kStartThreads);
    for (int c = 0; c < nch; ++c) {
      if (ok) ok = mbar_wait(&xfull[c % SX], (c / SX) & 1, p.wait_limit, abort_flag);
      if (ok && c + 1 < nch && c + 1 >= NB)
        ok = mbar_wait(&bufdone[(c + 1) % NB], ((c + 1 - NB) / NB) & 1, p.wait_limit, abort_flag);
      if (ok && c + 2 < nch) ok = mbar_wait(&wfull[(c + 2) % SW], ((c + 2) / SW) & 1, p.wait_limit, abort_flag);
      __syncwarp();
      named_bar_sync(kChunkBarrier, C::kBarThreads);
      // chunks up to c+1 are converted now
      if (lane == 0) {
        if (c == 0) mbar_arrive(&wempty[0]);
        if (c + 1 < nch) mbar_arrive(&wempty[(c + 1) % SW]);
      }
    }
  } else if (warp >= kDqWarp0) {
    const int d = warp - kDqWarp0;
    const int tile = d / C::kGroupWarps;        // the k tile of each chunk this warp converts
    const int rb = (d / 4) % RB;                // row block
    const int q = warp & 3;                     // TMEM lane quarter of this warp
    const int c4 = lane & 3;                    // this thread's columns: c4, c4+4, ... (k pairs 4i + c4)
    const uint32_t trow = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + kACol + 32u * (tile * RB + rb);
    // Software-pipelined by one chunk: the stores of chunk c are issued, then
    // chunk c+1 is loaded and converted in registers while they complete, and
    // only then does the warp wait for them and take the barrier.  a[0..15]
    // are TMEM lanes 32q + (0..15), a[16..31] lanes 32q + (16..31), each in the
    // 16x128b register order: a[16h + 2i + w] is channel 32q + 16h + lane/4 + 8w,
    // column 4i + c4.
    uint32_t a[32];
    // This warp's tile of chunk c, loaded from its weight stage (landed):
    // codes of channels 32q + lane/4 + 8w (w = 0..3) at k pairs 4i + c4, i =
    // 0..3 in w0 and 4..7 in w1; this 64-channel group's (scale, min) pairs
    // for those k pairs, unit u holding i = 2u and 2u+1.
    q4::BlockConverter<FMT> cv;
    auto load = [&](int c) {
      cv.load(wring + (c % SW) * C::kWStage + (rb * KT + tile) * kTileBytes, q, lane);
    };
    auto convert = [&]() { cv.convert(a, q, lane); };
    auto mine = [&](int c) { return tile < min(KT, nk - KT * c); };   // a ragged last chunk has one tile
    // The sync warp has seen the weights of chunks 0 and 1 land before this
    // barrier, and before chunk barrier c those of chunk c+2 and TMEM buffer
    // (c+1) % NB free.
    named_bar_sync(kStartBarrier, C::kStartThreads);
    if (nch > 0 && mine(0)) {
      load(0);
      convert();
    }
    for (int c = 0; c < nch; ++c) {
      const int b = c % NB;
      // chunk c+1's loads go out before chunk c's stores: a load queued
      // behind a tensor-memory store waits for it
      const bool next = c + 1 < nch && mine(c + 1);
      if (next) load(c + 1);
      if (mine(c)) {
        tc_fence_after();
        tmem_st_16x128b_x8(trow + b * C::kBufCols, a);
        tmem_st_16x128b_x8(trow + (16u << 16) + b * C::kBufCols, a + 16);
      }
      if (next) convert();
      tmem_st_wait();
      tc_fence_before();
      named_bar_sync(kChunkBarrier, C::kBarThreads);
    }
  }

  // ---- epilogue: TMEM lane = channel, column rb*kAcc + m = sequence m ---------------
  const bool epi = warp >= kDqWarp0 && warp < kDqWarp0 + 4 * RB;
  const int erb = (warp - kDqWarp0) >> 2;
  const int q = warp & 3;
  constexpr int NCH = RB * BNC;                 // channels of the tile
  bool ok = true;
  if (epi) {
    ok = mbar_wait(done, 0, p.wait_limit, abort_flag);
    if (!ok) {
      // the MMA warp always commits `done`: wait for its MMAs to finish
      // before touching or freeing the tensor memory they write
      volatile int dummy = 0;
      mbar_wait(done, 0, kDrainLimit, &dummy);
    }
    tc_fence_after();
    ok = ok && !*abort_flag;
  }
  griddep_wait();   // Y, the residual and the workspace belong to the stream order from here on
  const uint32_t tlane = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + erb * C::kAcc;
  const int lch = erb * BNC + 32 * q + lane;    // this lane's channel in the tile

  if (p.splits == 1) {
    if (epi) {
      const int ch = n0 + lch;
#pragma unroll 1
      for (int c0 = 0; c0 < BT && c0 < p.M; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tlane + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int m = c0 + e;
          if (m < p.M && ok) {
            float y = __uint_as_float(v[e]);
            if (p.R) y += __half2float(p.R[static_cast<size_t>(m) * p.ldr + ch]);
            if (p.relu) y = fmaxf(y, 0.0f);
            p.Y[static_cast<size_t>(m) * p.ldy + ch] = __float2half_rn(y);
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem_base, C::kTmemCols);
    }
    return;
  }

  // K splits: each split stages its partial, [M][NCH] fp32, in the drained
  // rings; the cluster's ranks (= splits) then share the rows of Y, each
  // summing every split's partial of its rows in split order over
  // distributed shared memory.
  float* stage = reinterpret_cast<float*>(xring);   // the rings are free: every load and MMA is done
  if (epi) {
#pragma unroll 1
    for (int c0 = 0; c0 < BT && c0 < p.M; c0 += 32) {
      uint32_t v[32];
      tmem_ld_32x32b_x32(tlane + c0, v);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (c0 + e < p.M) stage[(c0 + e) * NCH + lch] = ok ? __uint_as_float(v[e]) : 0.0f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
  cluster_sync();   // every split's partial is staged
  {
    // rank r reduces rows r, r + S, ... (S = splits): each item is four
    // consecutive channels of one row, read from every split's partial
    // (16 bytes each, all in flight at once) and summed in split order
    const int S = p.splits;
    const int r = static_cast<int>(cluster_ctarank());
    const int rows = (p.M - r + S - 1) / S;
    constexpr int kQuads = NCH / 4;
    for (int it = threadIdx.x; it < rows * kQuads; it += C::kThreads) {
      const int m = r + S * (it / kQuads), c = 4 * (it % kQuads);
      const float* item = stage + m * NCH + c;   // the same offset in every split's shared memory
      float4 v[kMaxSplits];
#pragma unroll
      for (int s = 0; s < kMaxSplits; ++s)
        if (s < S) v[s] = ld_shared_cluster_v4(mapa_shared(item, s));
      float4 y = v[0];
#pragma unroll
      for (int s = 1; s < kMaxSplits; ++s)
        if (s < S) {
          y.x += v[s].x;
          y.y += v[s].y;
          y.z += v[s].z;
          y.w += v[s].w;
        }
      const int ch = n0 + c;
      if (p.R) {
        const uint2 rr = *reinterpret_cast<const uint2*>(p.R + static_cast<size_t>(m) * p.ldr + ch);
        const float2 r01 = __half22float2(*reinterpret_cast<const __half2*>(&rr.x));
        const float2 r23 = __half22float2(*reinterpret_cast<const __half2*>(&rr.y));
        y.x += r01.x;
        y.y += r01.y;
        y.z += r23.x;
        y.w += r23.y;
      }
      if (p.relu) {
        y.x = fmaxf(y.x, 0.0f);
        y.y = fmaxf(y.y, 0.0f);
        y.z = fmaxf(y.z, 0.0f);
        y.w = fmaxf(y.w, 0.0f);
      }
      const __half2 y01 = __floats2half2_rn(y.x, y.y), y23 = __floats2half2_rn(y.z, y.w);
      *reinterpret_cast<uint2*>(p.Y + static_cast<size_t>(m) * p.ldy + ch) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&y01), *reinterpret_cast<const uint32_t*>(&y23));
    }
  }
  cluster_sync();   // no CTA leaves while another may still read its partial
}

template <int BT, int RB, int FMT>
fg_status launch_ts(TsParams& p, cudaStream_t st) {
  using C = TsCfg<BT, RB, FMT>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(gemm_q4ts_kernel<BT, RB, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kTotal) !=
        cudaSuccess)
      return check_launch("gemm_q4ts smem attribute");
    attr_set[dev] = true;
  }
  Trace tr(KC_GEMM_Q4DEC, st);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.n_tiles * p.splits));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kTotal;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;   // the K splits of a channel tile
  attr[1].val.clusterDim.x = static_cast<unsigned>(p.splits);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, gemm_q4ts_kernel<BT, RB, FMT>, p) != cudaSuccess)
    return check_launch("gemm_q4ts_kernel (launch)");
  return check_launch("gemm_q4ts_kernel");
}

int bt_for(int64_t M) { return M <= 32 ? 32 : (M <= 64 ? 64 : (M <= 128 ? 128 : 256)); }

// One row block per CTA: measured at b = 64, two CTAs of 128 channels per SM
// beat one of 256 (the X tile is re-read twice as often, but the two CTAs'
// pipelines overlap each other's stalls).
int rb_for(const GemmArgs&) { return 1; }

// Split count: K is cut so that the CTAs fill the GPU's slots (one per SM
// with two row blocks, two per SM with one) with the fewest waves of per-CTA
// k tiles, plus a charge per split for the cluster's reduction of its
// partial.  At most kMaxSplits (one portable cluster).  Depends on the shape
// only.
int splits_for(int64_t M, int64_t N, int64_t K, int rb) {
  const int64_t tiles = N / (BNC * rb), ktiles = K / BK;
  const int64_t slots = (rb == 1 && M <= 128 ? 2 : 1) * static_cast<int64_t>(num_sms());
  int64_t best = 1;
  double best_cost = 1e30;
  for (int64_t s = 1; s <= kMaxSplits && s <= ktiles / 2; ++s) {
    const int64_t waves = (tiles * s + slots - 1) / slots;
    const double cost = static_cast<double>(waves) * ((ktiles + s - 1) / s) + (s > 1 ? 2.0 + 0.5 * s : 0.0);
    if (cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return static_cast<int>(best);
}

}  // namespace

size_t gemm_q4ts_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }   // splits reduce in the cluster

bool gemm_q4ts_supported(const GemmArgs& a) {
  if (a.dtype != FG_F16 || !a.quant || a.M < 1 || a.M > 256 || a.K % BK) return false;
  for (int i = 0; i < a.nseg; ++i) {
    const WSeg& s = a.seg[i];
    if (!s.packed || s.N % BNC || !aligned(s.packed, 16)) return false;
    if (s.packed_format != a.seg[0].packed_format) return false;
    if (s.packed_format != FG_PACK_EXACT && s.packed_format != FG_PACK_F16META) return false;
  }
  if ((a.ldx * 2) % 16 || !aligned(a.X, 16)) return false;
  if (a.ldy % 4 || !aligned(a.Y, 8) || (a.R && (a.ldr % 4 || !aligned(a.R, 8)))) return false;
  return true;
}

fg_status gemm_q4ts(const GemmArgs& a, void* ws, size_t ws_bytes, cudaStream_t st) {
  (void)ws;   // the K splits reduce inside their cluster: no workspace
  (void)ws_bytes;
  TsParams p;
  memset(&p, 0, sizeof(p));
  const int bt = bt_for(a.M);
  const int rb = rb_for(a);
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.nseg = a.nseg;
  if (!tc_make_map(&p.mapX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.X, a.K, a.M, a.ldx * 2, BK, bt,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return fail(FG_ERR_CUDA, "tensor map for X");
  for (int i = 0; i < a.nseg; ++i) {
    p.seg_n0[i] = static_cast<int>(a.seg[i].n0);
    p.wp[i] = a.seg[i].packed;
  }
  p.seg_n0[a.nseg] = static_cast<int>(a.N);
  p.n_tiles = static_cast<int>(a.N / (BNC * rb));
  {
    const int ktiles = static_cast<int>(a.K / BK);
    const int want = splits_for(a.M, a.N, a.K, rb);
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
  p.wait_limit = wait_limit();
  if (a.seg[0].packed_format == FG_PACK_F16META) {
    switch (bt) {
      case 32: return launch_ts<32, 1, FG_PACK_F16META>(p, st);
      case 64: return launch_ts<64, 1, FG_PACK_F16META>(p, st);
      case 128: return launch_ts<128, 1, FG_PACK_F16META>(p, st);
      default: return launch_ts<256, 1, FG_PACK_F16META>(p, st);
    }
  }
  switch (bt) {
    case 32: return launch_ts<32, 1, FG_PACK_EXACT>(p, st);
    case 64: return launch_ts<64, 1, FG_PACK_EXACT>(p, st);
    case 128: return launch_ts<128, 1, FG_PACK_EXACT>(p, st);
    default: return launch_ts<256, 1, FG_PACK_EXACT>(p, st);
  }
}

fg_status pack_weight(const uint8_t* codes, const float* mins, const float* scales, int64_t K, int64_t N,
                      int format, uint8_t* packed, cudaStream_t st) {
  if (K == 0 || N == 0) return FG_OK;
  Trace tr(KC_PACK, st);
  constexpr int kT = 256;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
  const int64_t words = N * (K / 8), pairs = (N / 64) * (K / 2);
  pack_codes_kernel<<<static_cast<unsigned>(std::min<int64_t>((words + kT - 1) / kT, cap)), kT, 0, st>>>(
      codes, K, N, tile_bytes(format), packed);
  const fg_status sc = check_launch("pack_codes_kernel");
  if (sc != FG_OK) return sc;
  trace_extra_launch();
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>((pairs + kT - 1) / kT, cap));
  if (format == FG_PACK_F16META)
    pack_pairs_f16_kernel<<<grid, kT, 0, st>>>(mins, scales, K, N, packed);
  else
    pack_pairs_f32_kernel<<<grid, kT, 0, st>>>(mins, scales, K, N, packed);
  return check_launch("pack_pairs_kernel");
}

size_t pack_weight_bytes(int64_t K, int64_t N, int format) {
  return static_cast<size_t>(K / BK) * static_cast<size_t>(N / BNC) * tile_bytes(format);
}

}  // namespace fg
