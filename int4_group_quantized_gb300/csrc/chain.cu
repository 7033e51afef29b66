// Decode products of one layer-step in one persistent launch (FlexGen notes,
// "4. 卸载策略": zig-zag block, one read of a layer's weights serves every
// sequence of the block; "背景知识": the decode products t w_Q|w_K|w_V,
// t_Out = (..) w_O + t, relu(t_Out w_1), (..) w_2 + t_Out; "5. 近似方法":
// weights stored in 4-bit groups of 64 along the output channel, converted
// back to FP16 before compute).
//
// A chain is up to four products run back to back in one grid of one CTA per
// SM, each product's X either an input of the launch or the output of the
// product before it (e.g. w_O, w_1, w_2 of layer i and w_Q|w_K|w_V of layer
// i+1).  Each product's work -- (128-channel tile, 128-k chunk) units, tile
// major -- is cut into equal contiguous ranges, one per CTA ("stream-K"), so
// every CTA streams the same share of every weight and there is no wave
// quantisation and no separate split-sum launch.  A CTA's range covers the
// end of one tile, whole tiles, and the start of another: each piece is
// summed in a tensor-memory accumulator; a tile covered by one CTA gets its
// epilogue at once, otherwise every contributor writes its fp32 partial to
// its own workspace slot and the last to arrive (a per-tile counter) sums
// all of them in contributor order -- deterministic whoever is last --
// applies the epilogue and publishes the tile with a release flag.  The next
// product's X chunk k is exactly tile k of the product before it; the CTA
// that needs it waits on that flag (acquire, bounded) before its TMA load.
// Weights never wait: the weight copies of the next product stream while the
// current one finishes.
//
// Inside a CTA (384 threads, 256 TMEM columns, two CTAs per SM whose
// pipelines hide each other's stalls): warp 0 issues the weight copies (one
// 2-block bulk copy per chunk), warp 2 the X copies (after the flags), warp 3
// takes every mbarrier wait for the warps of the chunk barrier, warp 1 owns
// TMEM and issues the MMAs, warps 4..11 convert weights into TMEM (one block
// of the chunk per set of four, the BlockConverter register order).  The main
// loop runs in lockstep chunks: converting warps, sync warp and MMA warp meet
// at one named barrier per chunk, and the MMA warp issues the chunk's MMAs
// right after it.  A piece is summed in one accumulator; when it ends, the
// first four converting warps (one per TMEM lane quarter) drain it before the
// next chunk barrier -- the next piece's first MMAs overwrite it -- and run
// the piece's epilogue or its share of the tile's fixup.
//
// Every wait is bounded (fg_set_wait_limit): a wait that gives up raises the
// device error word and makes its role skip work, never a barrier; before the
// CTA leaves, its copies and MMAs in flight have completed and its tensor
// memory is freed.  Named barriers: the chunk barrier is taken once per chunk
// by the MMA, sync and 8 converting warps; the start barrier once by the sync
// and converting warps; the epilogue barrier the same number of times per
// piece by the 4 draining warps (the branch between its counts is decided
// once and broadcast through shared memory).
#include <cudaTypedefs.h>
#include <string.h>

#include <algorithm>

#include "fg_internal.cuh"
#include "q4_convert.cuh"
#include "q4_dev.cuh"
#include "tc_ptx.cuh"

namespace fg {

bool tc_make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

namespace {

using namespace tc;

constexpr int BK = 64;                 // k per block / MMA tile
constexpr int BNC = 128;               // channels per tile (the MMA's M)
constexpr int CK = 128;                // k per chunk: two blocks
constexpr int kThreads = 384;
constexpr int kCtasPerSm = 2;
constexpr int kConvWarp0 = 4;                       // 8 converting warps
constexpr int kChunkThreads = 64 + 8 * 32;          // MMA warp, sync warp, converters
constexpr int kStartThreads = 32 + 8 * 32;          // sync warp, converters
constexpr int kSyncWarp = 3;
constexpr uint32_t kChunkBar = 1, kStartBar = 2, kEpiBar = 3;
constexpr uint32_t kProducerSleepNs = 100;
constexpr uint32_t kFlagSleepNs = 64;
constexpr uint32_t kEpiSleepNs = 200;

struct ChainProduct {
  const uint8_t* wp[3];     // decode copy of each weight segment
  int seg_n0[4];            // segment column offsets, seg_n0[nseg] = N
  int nseg;
  int N, K;
  __half* Y;
  int ldy;
  const __half* R;          // residual [M][ldr] or null
  int ldr;
  int r_prod;               // product of this chain that wrote R, or -1
  int relu;
  int x_prod;               // product of this chain that writes X, or -1 (an input)
  unsigned* ready;          // [N/128] tile published (1) -- zero before the launch
  unsigned* cnt;            // [N/128] contributors arrived -- zero before the launch
  float* part;              // [N/128 + G - 1][M][128] fp32 partial slots
};

struct ChainParams {
  CUtensorMap mapX[kMaxChain];
  ChainProduct pr[kMaxChain];
  int np;
  int M;
  int G;                    // CTAs
  unsigned* err;
  uint32_t wait_limit;
};

// ---- the partition (identical on the host: chain_owner) -------------------------
// CTA c owns units [U c / G, U (c+1) / G) of a product with U units; unit u
// belongs to CTA floor(((u + 1) G - 1) / U).  U G stays below 2^31 (U <= 2^16
// units of 128 x 128 weights, G <= 256), so 32-bit arithmetic is exact.
__device__ __forceinline__ void cta_range(int U, int c, int G, int& u0, int& u1) {
  u0 = U * c / G;
  u1 = U * (c + 1) / G;
}
__device__ __forceinline__ int owner(int u, int U, int G) { return ((u + 1) * G - 1) / U; }

__device__ __forceinline__ uint32_t ld_acquire(const unsigned* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Returns the old value; acquire and release at GPU scope.  After a CTA
// barrier, one thread's release orders every write the barrier's threads
// made before it, and its acquire orders their reads after the next barrier.
__device__ __forceinline__ uint32_t atom_add_acq_rel(unsigned* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// Waits until *flag != 0 (acquire), polling at most `limit` times.
__device__ __forceinline__ bool wait_flag(const unsigned* flag, uint32_t limit, volatile int* abort) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (ld_acquire(flag) != 0) return true;
    if ((i & 255u) == 255u && *abort) return false;
    __nanosleep(kFlagSleepNs);
  }
  *abort = 1;
  return false;
}

// The piece of a CTA's range that ends at a chunk: tile n of product p,
// this CTA's contributor slot and the tile's contributor count.
struct Piece {
  int p, n, first, J;
  int dense;
  int index;   // the piece's number in this CTA (parity of its accumulator phase)
  int ended;   // the chunk that wrote this record ends the piece
};

// Drains the accumulator once the MMAs of the piece just ended are done and
// runs its epilogue (J == 1) or writes this CTA's partial and, for the last
// contributor to arrive, the tile's fixup; then publishes the tile.  Run by
// the four warps of TMEM lane quarters q = 0..3 (tid = 0..127); a call of its
// own, outside the converting loop's registers: it runs once per piece.
constexpr int chain_min(int a, int b) { return a < b ? a : b; }

template <int BT, int FMT>
struct ChainCfg {
  static constexpr int kBB = q4::block_bytes(FMT);   // one 128 x 64 weight block
  static constexpr int kWStage = 2 * kBB;            // a chunk's two blocks
  static constexpr int kXT = BT * BK * 2;            // one X tile, K-major, 128-byte swizzle
  static constexpr int kXStage = 2 * kXT;
  static constexpr int kAcc = BT < 32 ? 32 : BT;     // accumulator columns
  static constexpr int kACol = kAcc;                 // A buffers follow the accumulator
  static constexpr int kBufs = (256 - kACol) / 64;   // A buffers of 64 columns (a chunk)
  // X stages have their own release barriers (the MMA commit of the chunk
  // that read them), independent of the TMEM buffers
  static constexpr int kXStages = BT <= 32 ? 4 : 3;
  static constexpr int kSmemBudget = 108 * 1024;
  static constexpr int kWStages = chain_min(8, (kSmemBudget - kXStages * kXStage) / kWStage);
  static constexpr int kXBytes = kXStages * kXStage;
  static constexpr int kWBytes = kWStages * kWStage;
  static constexpr int kBarBytes = (2 * kXStages + 2 * kWStages + kBufs + 1) * 8 + 16 + 2 * sizeof(Piece);
  static constexpr int kTotal = 1024 + kXBytes + kWBytes + kBarBytes;
  static_assert(kBufs >= 3 && kWStages >= 3, "pipeline depth");
  static_assert(kXT % 1024 == 0, "X tiles stay 1024-byte aligned");
};

// Walks a CTA's chunks of every product of the chain in order, keeping the
// tile and chunk of the current unit (no division per chunk).
struct Walk {
  int p;                 // product
  int u, u0, u1;         // current unit, this product's range
  int cpt;               // chunks per tile of product p
  int tile, kc;          // u = tile * cpt + kc
  __device__ __forceinline__ void settle(const ChainParams& P, int cta) {
    while (p < P.np && u >= u1) {
      ++p;
      if (p < P.np) {
        const ChainProduct& q = P.pr[p];
        cpt = q.K / CK;
        cta_range((q.N / BNC) * cpt, cta, P.G, u0, u1);
        u = u0;
        tile = u0 / cpt;
        kc = u0 - tile * cpt;
      }
    }
  }
  __device__ __forceinline__ void start(const ChainParams& P, int cta) {
    p = -1;
    u = u1 = 0;
    settle(P, cta);
  }
  __device__ __forceinline__ void next(const ChainParams& P, int cta) {
    ++u;
    if (++kc == cpt) {
      kc = 0;
      ++tile;
    }
    settle(P, cta);
  }
  __device__ __forceinline__ bool first() const { return u == u0 || kc == 0; }
  __device__ __forceinline__ bool last() const { return u + 1 == u1 || kc + 1 == cpt; }
};

__device__ __forceinline__ int total_chunks(const ChainParams& P, int cta) {
  int n = 0;
  for (int p = 0; p < P.np; ++p) {
    int u0, u1;
    cta_range((P.pr[p].N / BNC) * (P.pr[p].K / CK), cta, P.G, u0, u1);
    n += u1 - u0;
  }
  return n;
}

template <int BT>
__device__ __forceinline__ void drain_piece(const ChainParams& P, const Piece pc, int q, int lane, int tid,
                                         uint32_t tmem_base, int cta, uint64_t* accfull, volatile int* abort_flag,
                                         volatile int* epi_last) {
  const int M = P.M;
    const ChainProduct& qp = P.pr[pc.p];
    bool ok = true;
    if (lane == 0) {
      ok = mbar_wait_sleep(accfull, static_cast<uint32_t>(pc.index & 1), P.wait_limit, abort_flag, kEpiSleepNs);
      if (!ok) {
        volatile int dummy = 0;   // the MMAs are always committed: let them finish first
        mbar_wait(accfull, static_cast<uint32_t>(pc.index & 1), kDrainLimit, &dummy);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    tc_fence_after();
    ok = ok && !*abort_flag;
    griddep_wait();   // Y, R and the partial slots belong to the stream order
    if (pc.J == 1 && qp.R && qp.r_prod >= 0) ok = ok && wait_flag(P.pr[qp.r_prod].ready + pc.n, P.wait_limit, abort_flag);
    const int ch = pc.n * BNC + 32 * q + lane;   // this thread's channel (= TMEM lane)
    float* mine = qp.part + static_cast<size_t>(pc.n + cta) * M * BNC + 32 * q + lane;
    const uint32_t ta = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
#pragma unroll 1
    for (int r0 = 0; r0 < BT; r0 += 16) {
      uint32_t r[16];
      tmem_ld_32x32b_x16(ta + r0, r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int m = r0 + e;
        if (m >= M) continue;
        const float v = __uint_as_float(r[e]);
        if (pc.J == 1) {
          float y = v;
          if (qp.R) y += __half2float(__ldcg(qp.R + static_cast<size_t>(m) * qp.ldr + ch));
          if (qp.relu) y = fmaxf(y, 0.0f);
          if (ok) qp.Y[static_cast<size_t>(m) * qp.ldy + ch] = __float2half_rn(y);
        } else {
          mine[m * BNC] = v;
        }
      }
    }
    tc_fence_before();   // the accumulator reads, before the barrier after which it is overwritten
    if (pc.J > 1) {
      named_bar_sync(kEpiBar, 128);
      if (tid == 0) *epi_last = atom_add_acq_rel(qp.cnt + pc.n, 1u) == static_cast<unsigned>(pc.J - 1);
      named_bar_sync(kEpiBar, 128);
      if (*epi_last == 0) return;   // the same for the four warps: no barrier below is skipped unevenly
      if (qp.R && qp.r_prod >= 0) ok = ok && wait_flag(P.pr[qp.r_prod].ready + pc.n, P.wait_limit, abort_flag);
      // The last to arrive sums the J partials in contributor order (the
      // same sum whichever CTA is last).  Thread tid takes channels
      // 4 (tid % 32) .. +3 of rows m = tid / 32 + 4 i: 16-byte loads, each
      // warp reading whole 512-byte rows, two rows at a time, the next
      // contributor's loads in flight while the current one is added.
      const int c4 = 4 * (tid & 31), m0 = tid >> 5;
      const int U = (qp.N / BNC) * (qp.K / CK), cpt = qp.K / CK;
      constexpr int kRows = BT / 4;          // rows per thread
      constexpr int kGrp = 2;
#pragma unroll 1
      for (int g0 = 0; g0 < kRows; g0 += kGrp) {
        float4 acc[kGrp], b0[kGrp], b1[kGrp];
        auto slot_of = [&](int k) {
          const int c = pc.dense ? pc.first + k : owner(pc.n * cpt + k, U, P.G);
          return reinterpret_cast<const float4*>(qp.part + static_cast<size_t>(pc.n + c) * M * BNC + c4);
        };
        auto fetch = [&](float4 (&dst)[kGrp], const float4* src) {
#pragma unroll
          for (int i = 0; i < kGrp; ++i) {
            const int m = m0 + 4 * (g0 + i);
            dst[i] = m < M ? __ldcg(src + m * (BNC / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        };
        auto add = [&](const float4 (&src)[kGrp]) {
#pragma unroll
          for (int i = 0; i < kGrp; ++i) {
            acc[i].x += src[i].x;
            acc[i].y += src[i].y;
            acc[i].z += src[i].z;
            acc[i].w += src[i].w;
          }
        };
        fetch(acc, slot_of(0));
        fetch(b0, slot_of(1));
#pragma unroll 1
        for (int k = 1; k < pc.J; k += 2) {
          if (k + 1 < pc.J) fetch(b1, slot_of(k + 1));
          add(b0);
          if (k + 1 < pc.J) {
            if (k + 2 < pc.J) fetch(b0, slot_of(k + 2));
            add(b1);
          }
        }
#pragma unroll
        for (int i = 0; i < kGrp; ++i) {
          const int m = m0 + 4 * (g0 + i);
          if (m >= M) continue;
          const int chq = pc.n * BNC + c4;
          float y[4] = {acc[i].x, acc[i].y, acc[i].z, acc[i].w};
          if (qp.R) {
            const uint2 rr = __ldcg(reinterpret_cast<const uint2*>(qp.R + static_cast<size_t>(m) * qp.ldr + chq));
            const float2 r01 = __half22float2(*reinterpret_cast<const __half2*>(&rr.x));
            const float2 r23 = __half22float2(*reinterpret_cast<const __half2*>(&rr.y));
            y[0] += r01.x;
            y[1] += r01.y;
            y[2] += r23.x;
            y[3] += r23.y;
          }
          if (qp.relu) {
#pragma unroll
            for (int e = 0; e < 4; ++e) y[e] = fmaxf(y[e], 0.0f);
          }
          const __half2 y01 = __floats2half2_rn(y[0], y[1]), y23 = __floats2half2_rn(y[2], y[3]);
          if (ok)
            *reinterpret_cast<uint2*>(qp.Y + static_cast<size_t>(m) * qp.ldy + chq) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&y01), *reinterpret_cast<const uint32_t*>(&y23));
        }
      }
    }
    // publish the tile: the release after the barrier orders every thread's stores of it
    named_bar_sync(kEpiBar, 128);
    if (tid == 0) {
      if (pc.J > 1) qp.cnt[pc.n] = 0;   // every contributor has arrived: ready for the next launch
      st_release(qp.ready + pc.n, 1u);
    }
}

template <int BT, int FMT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) chain_kernel(const __grid_constant__ ChainParams P) {
  using C = ChainCfg<BT, FMT>;
  constexpr int NB = C::kBufs, SX = C::kXStages, SW = C::kWStages;
  constexpr uint32_t kIdesc = idesc_f16(128, BT, 0, 0);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* xring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wring = xring + C::kXBytes;
  uint64_t* xfull = reinterpret_cast<uint64_t*>(wring + C::kWBytes);
  uint64_t* xempty = xfull + SX;       // X stage read by its chunk's MMAs
  uint64_t* wfull = xempty + SX;
  uint64_t* wempty = wfull + SW;
  uint64_t* bufdone = wempty + SW;     // MMAs of the chunk in TMEM buffer b completed
  uint64_t* accfull = bufdone + NB;    // the piece in the accumulator is summed (one phase per piece)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_last = abort_flag + 1;
  // the piece record of chunk g, in slot g % 2: written by the MMA warp before
  // chunk barrier g, read by the draining warps after it
  Piece* pinfo = reinterpret_cast<Piece*>(reinterpret_cast<uint8_t*>(tmem_slot) + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int nch = total_chunks(P, cta);

  griddep_launch();

  if (threadIdx.x == 0) {
    for (int i = 0; i < SX; ++i) {
      mbar_init(&xfull[i], 1);
      mbar_init(&xempty[i], 1);        // the MMA commit
    }
    for (int i = 0; i < SW; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], 1);
    }
    for (int i = 0; i < NB; ++i) mbar_init(&bufdone[i], 1);
    mbar_init(accfull, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 256);
  if (warp == 2 && lane == 0)
    for (int p = 0; p < P.np; ++p) tma_prefetch_desc(&P.mapX[p]);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---- weight copies: independent of every flag, so they run ahead ----------------
    if (lane == 0) {
      Walk w;
      w.start(P, cta);
      int issued = 0;
      for (int g = 0; g < nch; ++g, w.next(P, cta)) {
        const int s = g % SW;
        if (!mbar_wait_sleep(&wempty[s], static_cast<uint32_t>((g / SW) & 1) ^ 1u, P.wait_limit, abort_flag,
                             kProducerSleepNs))
          break;
        const ChainProduct& q = P.pr[w.p];
        const int n0 = w.tile * BNC;
        int seg = 0;
        while (seg + 1 < q.nseg && n0 >= q.seg_n0[seg + 1]) ++seg;
        const size_t run = static_cast<size_t>(q.K / BK) * C::kBB;   // the k blocks of one tile
        const uint8_t* src = q.wp[seg] + static_cast<size_t>((n0 - q.seg_n0[seg]) / BNC) * run +
                             static_cast<size_t>(w.kc) * C::kWStage;
        mbar_expect_tx(&wfull[s], C::kWStage);
        bulk_load(wring + s * C::kWStage, src, C::kWStage, &wfull[s]);
        ++issued;
      }
      for (int g = issued > SW ? issued - SW : 0; g < issued; ++g) {   // nothing in flight at exit
        volatile int dummy = 0;
        mbar_wait(&wfull[g % SW], static_cast<uint32_t>((g / SW) & 1), kDrainLimit, &dummy);
      }
      if (*abort_flag) atomicOr(P.err, DEV_ERR_WAIT_TIMEOUT);
    }
    __syncwarp();   // the warp reaches the CTA barrier below converged
  } else if (warp == 2) {
    // ---- X copies: chunk k of a product's X is tile k of the product before it -------
    if (lane == 0) {
      griddep_wait();   // inputs, flags and counters belong to the stream order from here on
      Walk w;
      w.start(P, cta);
      int issued = 0;
      for (int g = 0; g < nch; ++g, w.next(P, cta)) {
        const int s = g % SX;
        // the MMAs of chunk g - SX, the last to read stage s, have completed
        if (!mbar_wait_sleep(&xempty[s], static_cast<uint32_t>((g / SX) & 1) ^ 1u, P.wait_limit, abort_flag,
                             kProducerSleepNs))
          break;
        const ChainProduct& q = P.pr[w.p];
        const int kc = w.kc;
        if (q.x_prod >= 0) {
          if (!wait_flag(P.pr[q.x_prod].ready + kc, P.wait_limit, abort_flag)) break;
          fence_proxy_async_global();   // the acquired tile, to the TMA reads that follow
        }
        mbar_expect_tx(&xfull[s], C::kXStage);
        for (int t = 0; t < 2; ++t)
          tma_load_2d(xring + s * C::kXStage + t * C::kXT, &P.mapX[w.p], kc * CK + t * BK, 0, &xfull[s]);
        ++issued;
      }
      for (int g = issued > SX ? issued - SX : 0; g < issued; ++g) {
        volatile int dummy = 0;
        mbar_wait(&xfull[g % SX], static_cast<uint32_t>((g / SX) & 1), kDrainLimit, &dummy);
      }
      if (*abort_flag) atomicOr(P.err, DEV_ERR_WAIT_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMAs: every lane takes the chunk barrier, lane 0 issues ---------------------
    Walk w;
    w.start(P, cta);
    int piece = -1;
    Piece pc = {0, 0, 0, 0, 0, -1, 0};
    for (int g = 0; g < nch; ++g, w.next(P, cta)) {
      const bool first = w.first(), last = w.last();
      if (first) {
        ++piece;
        const ChainProduct& qp = P.pr[w.p];
        const int cpt = qp.K / CK, U = (qp.N / BNC) * cpt;
        pc.p = w.p;
        pc.n = w.tile;
        pc.first = owner(w.tile * cpt, U, P.G);
        pc.dense = U >= P.G;
        // the tile's contributors, in order: with at least as many units as
        // CTAs every CTA from the owner of the tile's first unit to the owner
        // of its last; with fewer, every CTA holds at most one unit, and the
        // contributors are the owners of the tile's units
        pc.J = pc.dense ? owner((w.tile + 1) * cpt - 1, U, P.G) - pc.first + 1 : cpt;
        pc.index = piece;
      }
      pc.ended = last;
      if (lane == 0) pinfo[g & 1] = pc;
      named_bar_sync(kChunkBar, kChunkThreads);   // chunk g in TMEM, its X landed, the accumulator drained
      if (lane == 0) {
        tc_fence_after();
        const int b = g % NB;
        if (!*abort_flag) {
          const uint64_t d0 = smem_desc_sw128(smem_u32(xring + (g % SX) * C::kXStage), 16, 1024);
          const uint32_t ta = tmem_base + C::kACol + b * 64;
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_f16_ts(tmem_base, ta + 32u * t + 8u * kk, d0 + ((t * C::kXT + kk * 32) >> 4), kIdesc,
                         (first && t == 0 && kk == 0) ? 0u : 1u);
        }
        mma_commit(&bufdone[b]);
        mma_commit(&xempty[g % SX]);
        if (last) mma_commit(accfull);
      }
      __syncwarp();
    }
  } else if (warp == kSyncWarp) {
    // ---- waits on behalf of the warps that take the chunk barrier ----------------------
    // Before chunk barrier g: chunk g's X, TMEM buffer (g+1) % NB free (the MMAs
    // of chunk g+1-NB done) and the weights of chunk g+2 landed.  After it:
    // the weight stages converted by then are released.
    bool ok = nch == 0 || (mbar_wait(&wfull[0], 0, P.wait_limit, abort_flag) &&
                           (nch < 2 || mbar_wait(&wfull[1 % SW], (1 / SW) & 1, P.wait_limit, abort_flag)));
    named_bar_sync(kStartBar, kStartThreads);
    for (int g = 0; g < nch; ++g) {
      if (ok) ok = mbar_wait(&xfull[g % SX], static_cast<uint32_t>((g / SX) & 1), P.wait_limit, abort_flag);
      if (ok && g + 1 < nch && g + 1 >= NB)
        ok = mbar_wait(&bufdone[(g + 1) % NB], static_cast<uint32_t>(((g + 1 - NB) / NB) & 1), P.wait_limit,
                       abort_flag);
      if (ok && g + 2 < nch)
        ok = mbar_wait(&wfull[(g + 2) % SW], static_cast<uint32_t>(((g + 2) / SW) & 1), P.wait_limit, abort_flag);
      __syncwarp();
      named_bar_sync(kChunkBar, kChunkThreads);
      if (lane == 0) {
        if (g == 0) mbar_arrive(&wempty[0]);
        if (g + 1 < nch) mbar_arrive(&wempty[(g + 1) % SW]);
      }
    }
  } else {
    // ---- conversion of the weights into TMEM; the first four warps also drain -----------
    const int d = warp - kConvWarp0;
    const int t = d >> 2;                 // which block of the chunk
    const int q = warp & 3;               // TMEM lane quarter
    const bool drains = d < 4;            // one warp per lane quarter
    const int tid = threadIdx.x - 32 * kConvWarp0;   // 0..127 for the draining warps
    const uint32_t trow = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + C::kACol + 32u * t;
    const int M = P.M;
    q4::BlockConverter<FMT> cv;
    uint32_t a[32];

    // Drains the accumulator once the MMAs of the piece just ended are done and
    // runs its epilogue (J == 1) or writes this CTA's partial and, for the last
    // contributor to arrive, the tile's fixup; then publishes the tile.
    named_bar_sync(kStartBar, kStartThreads);
    if (nch > 0) {
      cv.load(wring + t * C::kBB, q, lane);
      cv.convert(a, q, lane);
    }
    for (int g = 0; g < nch; ++g) {
      const bool next = g + 1 < nch;
      const uint32_t dst = trow + static_cast<uint32_t>(g % NB) * 64;
      // the record of chunk g-1 (written before chunk barrier g-1)
      const bool ended = drains && g > 0 && pinfo[(g - 1) & 1].ended;
      if (ended) {
        // chunk g's MMAs come after this chunk's barrier: drain the piece that
        // ended at chunk g-1 first (between the stores of chunk g and the
        // loads of chunk g+1, where neither holds registers)
        tc_fence_after();
        tmem_st_16x128b_x8(dst, a);
        tmem_st_16x128b_x8(dst + (16u << 16), a + 16);
        drain_piece<BT>(P, pinfo[(g - 1) & 1], q, lane, tid, tmem_base, cta, accfull, abort_flag, epi_last);
        if (next) cv.load(wring + ((g + 1) % SW) * C::kWStage + t * C::kBB, q, lane);
      } else {
        // the next chunk's loads go out before this chunk's stores
        if (next) cv.load(wring + ((g + 1) % SW) * C::kWStage + t * C::kBB, q, lane);
        tc_fence_after();
        tmem_st_16x128b_x8(dst, a);
        tmem_st_16x128b_x8(dst + (16u << 16), a + 16);
      }
      if (next) cv.convert(a, q, lane);
      tmem_st_wait();
      tc_fence_before();
      named_bar_sync(kChunkBar, kChunkThreads);
    }
    if (drains && nch > 0)   // the last piece always ends at the last chunk
      drain_piece<BT>(P, pinfo[(nch - 1) & 1], q, lane, tid, tmem_base, cta, accfull, abort_flag, epi_last);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 256);
  }
}

template <int BT, int FMT>
fg_status launch_chain(const ChainParams& P, cudaStream_t st, bool pdl) {
  using C = ChainCfg<BT, FMT>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(chain_kernel<BT, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kTotal) !=
        cudaSuccess)
      return check_launch("chain smem attribute");
    attr_set[dev] = true;
  }
  Trace tr(KC_GEMM_Q4DEC, st);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(P.G));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kTotal;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, chain_kernel<BT, FMT>, P) != cudaSuccess) return check_launch("chain_kernel (launch)");
  return check_launch("chain_kernel");
}

}  // namespace

int chain_owner(int64_t u, int64_t U, int G) { return static_cast<int>(((u + 1) * G - 1) / U); }

static_assert(kChainMaxCtas * 65536LL < (1LL << 31), "32-bit partition arithmetic");

int chain_ctas() { return std::min(kCtasPerSm * num_sms(), kChainMaxCtas); }

size_t chain_part_bytes(int64_t M, int64_t N) {
  return static_cast<size_t>(N / BNC + kChainMaxCtas - 1) * static_cast<size_t>(M) * BNC * sizeof(float);
}

size_t chain_ctrl_bytes(int64_t N) { return static_cast<size_t>(N / BNC) * 2 * sizeof(unsigned); }

bool chain_supported(const GemmArgs& a) {
  if (a.dtype != FG_F16 || !a.quant || a.M < 1 || a.M > 64 || a.K % CK || a.N % BNC) return false;
  if ((a.N / BNC) * (a.K / CK) > 65536) return false;   // the kernel's 32-bit partition arithmetic
  for (int i = 0; i < a.nseg; ++i) {
    const WSeg& s = a.seg[i];
    if (!s.packed || s.N % BNC || !aligned(s.packed, 16) || s.packed_format != a.seg[0].packed_format) return false;
    if (s.packed_format != FG_PACK_EXACT && s.packed_format != FG_PACK_F16META) return false;
  }
  if ((a.ldx * 2) % 16 || !aligned(a.X, 16)) return false;
  if (a.ldy % 8 || !aligned(a.Y, 16) || (a.R && (a.ldr % 8 || !aligned(a.R, 16)))) return false;
  return true;
}

fg_status chain_run(const ChainLink* links, int n, void* part_ws, size_t part_bytes, unsigned* ctrl,
                    size_t ctrl_bytes, bool ctrl_zeroed, cudaStream_t st) {
  if (n < 1 || n > kMaxChain) return fail(FG_ERR_ARG, "chain of %d products", n);
  ChainParams P;
  memset(&P, 0, sizeof(P));
  P.np = n;
  P.M = static_cast<int>(links[0].a.M);
  P.G = chain_ctas();
  P.err = device_error_word();
  if (!P.err) return fail(FG_ERR_CUDA, "device error word");
  P.wait_limit = wait_limit();
  char* part = static_cast<char*>(part_ws);
  size_t pused = 0, cused = 0;
  const int fmt = links[0].a.seg[0].packed_format;
  for (int i = 0; i < n; ++i) {
    const GemmArgs& a = links[i].a;
    if (!chain_supported(a) || a.M != P.M || a.seg[0].packed_format != fmt)
      return fail(FG_ERR_ARG, "product %d cannot join the chain", i);
    ChainProduct& q = P.pr[i];
    if (!tc_make_map(&P.mapX[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.X, a.K, a.M, a.ldx * 2, BK,
                     static_cast<uint32_t>(a.M <= 32 ? 32 : 64), CU_TENSOR_MAP_SWIZZLE_128B))
      return fail(FG_ERR_CUDA, "tensor map for X of product %d", i);
    for (int s = 0; s < a.nseg; ++s) {
      q.wp[s] = a.seg[s].packed;
      q.seg_n0[s] = static_cast<int>(a.seg[s].n0);
    }
    q.nseg = a.nseg;
    q.seg_n0[a.nseg] = static_cast<int>(a.N);
    q.N = static_cast<int>(a.N);
    q.K = static_cast<int>(a.K);
    q.Y = static_cast<__half*>(a.Y);
    q.ldy = static_cast<int>(a.ldy);
    q.R = static_cast<const __half*>(a.R);
    q.ldr = static_cast<int>(a.ldr);
    q.r_prod = links[i].r_prod;
    q.relu = a.relu;
    q.x_prod = links[i].x_prod;
    if (q.x_prod >= i || q.r_prod >= i) return fail(FG_ERR_ARG, "a chain product reads a later product");
    if (q.x_prod >= 0 && P.pr[q.x_prod].N != q.K) return fail(FG_ERR_SHAPE, "chain X width");
    if (q.r_prod >= 0 && (!q.R || P.pr[q.r_prod].N != q.N)) return fail(FG_ERR_SHAPE, "chain residual width");
    const size_t pb = chain_part_bytes(a.M, a.N), cb = chain_ctrl_bytes(a.N);
    if (pused + pb > part_bytes || cused + cb > ctrl_bytes) return fail(FG_ERR_WORKSPACE, "chain workspace");
    q.part = reinterpret_cast<float*>(part + pused);
    q.ready = ctrl + cused / sizeof(unsigned);
    q.cnt = q.ready + a.N / BNC;
    pused += (pb + 255) / 256 * 256;
    cused += cb;
  }
  if (!ctrl_zeroed) {
    if (cudaMemsetAsync(ctrl, 0, cused, st) != cudaSuccess) return check_launch("chain control reset");
  }
  const bool pdl = ctrl_zeroed;   // after a memset the launch keeps the full stream order
  if (fmt == FG_PACK_F16META)
    return P.M <= 32 ? launch_chain<32, FG_PACK_F16META>(P, st, pdl) : launch_chain<64, FG_PACK_F16META>(P, st, pdl);
  return P.M <= 32 ? launch_chain<32, FG_PACK_EXACT>(P, st, pdl) : launch_chain<64, FG_PACK_EXACT>(P, st, pdl);
}

size_t chain_workspace_bytes(const int64_t* N, int n, int64_t M) {
  size_t b = 0;
  for (int i = 0; i < n; ++i) b += (chain_part_bytes(M, N[i]) + 255) / 256 * 256;
  return b;
}

}  // namespace fg
