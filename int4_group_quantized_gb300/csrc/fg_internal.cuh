// Internal declarations shared by the libfg.so translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fg.h"

namespace fg {

// ---- host-side error reporting -------------------------------------------
// Records a printf-style detail for fg_last_error() and returns `s`.
fg_status fail(fg_status s, const char* fmt, ...);
// Maps cudaGetLastError() after a launch to FG_OK / FG_ERR_CUDA.
fg_status check_launch(const char* what);
// Return the status of `expr` when it is not FG_OK.
#define FG_TRY(expr)                 \
  do {                               \
    fg_status _s = (expr);           \
    if (_s != FG_OK) return _s;      \
  } while (0)

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t dtype_bytes(fg_dtype d) { return d == FG_F16 ? 2 : 4; }
// Number of SMs of the current device (cached per device).
int num_sms();
// Device address of the library's error word on the current device; kernels
// that run bounded waits OR an error code into it.
unsigned int* device_error_word();

enum DeviceError : unsigned int { DEV_ERR_WAIT_TIMEOUT = 1u };
// Polls a bounded wait makes before it gives up (fg_set_wait_limit), passed
// to every kernel that waits.  Waits for work that is already in flight (a
// copy issued, an MMA committed) use kDrainLimit instead: a CTA never leaves
// with its own copies or MMAs outstanding.
uint32_t wait_limit();
constexpr uint32_t kDrainLimit = 1u << 26;

// ---- launch tracing ----------------------------------------------------------
// Every kernel launch is bracketed by a Trace; while fg_profile_start() is
// active each launch gets a pair of CUDA events on its stream, accumulated per
// kernel class by fg_profile_stop().  A launch counter runs always.
enum KernelClass : int {
  KC_QUANTIZE = 0,
  KC_DEQUANT,
  KC_KV_STORE,
  KC_GEMM_SIMT,
  KC_GEMM_TC,
  KC_GEMM_REDUCE,
  KC_ATTN_DECODE,
  KC_ATTN_COMBINE,
  KC_ATTN_PREFILL,
  KC_GEMM_Q4DEC,
  KC_PACK,
  KC_ATTN_TOPK,
  KC_COUNT
};
constexpr int kProfilePhases = 4;
void trace_begin(int cls, cudaStream_t st);
void trace_end(int cls, cudaStream_t st);
// A second kernel launched inside a Trace scope, timed as part of that
// scope's launch (only the launch counter sees it).
void trace_extra_launch();
// The launch counter for kernels a CUDA graph runs (n per replay), and its
// correction for launches only recorded into a graph.
void count_launches(uint64_t n);
void count_launches_undo(uint64_t n);
bool profiling();   // fg_profile_start is active
struct Trace {
  int cls;
  cudaStream_t st;
  Trace(int c, cudaStream_t s) : cls(c), st(s) { trace_begin(c, s); }
  ~Trace() { trace_end(cls, st); }
};

// ---- weight operand of a product -----------------------------------------
// A product's B operand may be split into up to three matrices laid side by
// side along N (w_Q | w_K | w_V share one launch); each segment's N is a
// multiple of 64 and its columns start at `n0` in the output.
struct WSeg {
  const uint8_t* codes;
  const uint8_t* packed;   // the decode copy (fg_pack_weight) or null
  int packed_format;       // fg_pack_format of `packed`
  const float* mins;
  const float* scales;
  const void* dense;
  int64_t N;
  int64_t n0;
};

struct GemmArgs {
  const void* X;     // [M][K], row stride ldx (elements)
  int64_t ldx;
  int64_t M, K;
  WSeg seg[3];
  int nseg;
  int64_t N;         // total columns = sum of segment N
  void* Y;           // [M][N], row stride ldy
  int64_t ldy;
  const void* R;     // optional residual [M][N], row stride ldr
  int64_t ldr;
  int relu;
  int quant;         // 1: segments are Q4G64, 0: dense
  fg_dtype dtype;
};

// CUDA-core product (any M, fp16 or fp32).
fg_status gemm_simt(const GemmArgs& a, cudaStream_t st);
// Tensor-core product on dense fp16 weights (M >= 64), operands by TMA.
bool gemm_tc_supported(const GemmArgs& a);
fg_status gemm_tc(const GemmArgs& a, void* ws, size_t ws_bytes, cudaStream_t st);
size_t gemm_tc_workspace_bytes(int64_t M, int64_t N, int64_t K);
// Decode product on channel-major packed 4-bit weights for M <= 256 rows:
// the weights are dequantized straight into tensor memory (the MMA's A
// operand), so shared memory carries only codes, (min, scale) and X.
// K splits go through `ws` (gemm_q4ts_workspace_bytes).
bool gemm_q4ts_supported(const GemmArgs& a);
fg_status gemm_q4ts(const GemmArgs& a, void* ws, size_t ws_bytes, cudaStream_t st);
size_t gemm_q4ts_workspace_bytes(int64_t M, int64_t N, int64_t K);
// The decode copy of a [K][N] 4-bit weight read by gemm_q4ts (fg_pack_weight),
// in fg_pack_format `format`, and its size.
fg_status pack_weight(const uint8_t* codes, const float* mins, const float* scales, int64_t K, int64_t N,
                      int format, uint8_t* packed, cudaStream_t st);
size_t pack_weight_bytes(int64_t K, int64_t N, int format);

// Y = epilogue(X . W); chooses the kernel for the operands:
//   fp16, 4-bit weights with their decode copy, M <= 256: gemm_q4ts;
//   fp16, 4-bit weights without it, M >= 64: the weight converted back to
//     fp16 into the workspace, then gemm_tc;
//   fp16, dense weights, M >= 64: gemm_tc;
//   everything else (fp32, fewer than 64 rows without a decode copy): gemm_simt.
// `ws` (ws_bytes >= gemm_workspace_bytes) holds split-K partial sums and the
// converted weight where a path needs them; `packed` says whether every
// weight segment carries its decode copy.
fg_status gemm(const GemmArgs& a, void* ws, size_t ws_bytes, cudaStream_t st);
size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, fg_dtype dt, int quant, bool packed);

// ---- KV cache --------------------------------------------------------------
// Store K/V rows of `T` tokens per sequence at slots pos0..pos0+T-1.  The
// row of sequence bi, token ti starts at ksrc + (bi*T + ti)*ld (elements of
// the cache dtype), likewise for vsrc.
// write_back (4-bit fp16 cache): each source row is then overwritten with the
// values the cache restores, fp16(fmaf(q, scale, min)).
fg_status kv_store(const fg_kv& kv, const void* ksrc, const void* vsrc, int64_t ld, int64_t b,
                   int64_t T, int64_t pos0, cudaStream_t st, bool write_back = false);
// Causal prefill attention on tcgen05 over a Q|K|V buffer [b*s][ld] whose K
// and V columns hold the values the cache restores (kv_store with
// write_back): s a multiple of 128, head_dim 64 or 128, fp16.
bool prefill_attention_tc_supported(int64_t s, int32_t head_dim, fg_dtype dt);
fg_status prefill_attention_tc(const void* qkv, int64_t ld, int64_t b, int64_t s, int32_t heads, int32_t head_dim,
                               void* out, int64_t ldo, cudaStream_t st);

// ---- attention -------------------------------------------------------------
// Host-side argument checks of fg_decode_attention (no CUDA call).
fg_status check_decode_attention(const fg_kv* kv, const void* q, int64_t ldq, int64_t pos, const void* out,
                                 int64_t ldo);
// Decode: one query per (sequence, head) at slot pos over slots 0..pos.
// q: [b][ldq] (head h at columns h*d..), out: [b][ldo].  When knew/vnew are
// given ([b][ldnew] rows), the new token's K/V are first written to slot pos
// (fused into the attention launch on the tensor-core path).
fg_status decode_attention(const fg_kv& kv, const void* q, int64_t ldq, const void* knew,
                           const void* vnew, int64_t ldnew, int64_t b, int64_t pos, void* out,
                           int64_t ldo, void* ws, size_t ws_bytes, cudaStream_t st);
size_t decode_attention_workspace_bytes(int64_t b, int32_t heads, int32_t head_dim,
                                        int64_t capacity);
fg_status decode_attention_simt(const fg_kv& kv, const void* q, int64_t ldq, int64_t b,
                                int64_t pos, void* out, int64_t ldo, cudaStream_t st);
// Top-K sparse decode attention (one CTA per (sequence, head), no split):
// the keep largest scores of each query, ties to the lower index, weighted
// by the softmax over all tokens; knew/vnew as for decode_attention.  idx,
// when given, receives the kept slots [b][heads][min(keep, pos+1)] in
// ascending order.
fg_status check_decode_attention_topk(const fg_kv* kv, const void* q, int64_t ldq, int64_t pos, int64_t keep,
                                      const void* out, int64_t ldo, const int32_t* idx);
fg_status decode_attention_topk(const fg_kv& kv, const void* q, int64_t ldq, const void* knew, const void* vnew,
                                int64_t ldnew, int64_t pos, int64_t keep, void* out, int64_t ldo, int32_t* idx,
                                cudaStream_t st);
// Prefill: causal attention of s queries per sequence over slots 0..s-1.
// q: [b*s][ldq]; out: [b*s][ldo].  Tensor cores for a 4-bit fp16 cache,
// CUDA cores otherwise.
fg_status prefill_attention(const fg_kv& kv, const void* q, int64_t ldq, int64_t b, int64_t s,
                            void* out, int64_t ldo, cudaStream_t st);
fg_status prefill_attention_simt(const fg_kv& kv, const void* q, int64_t ldq, int64_t b, int64_t s,
                                 void* out, int64_t ldo, cudaStream_t st);

// ---- codec -----------------------------------------------------------------
fg_status quantize_rows(const void* x, fg_dtype dt, int64_t rows, int64_t cols, uint8_t* codes,
                        float* mins, float* scales, cudaStream_t st);
fg_status dequant_rows(const uint8_t* codes, const float* mins, const float* scales,
                       int64_t rows, int64_t cols, void* out, fg_dtype dt, cudaStream_t st);

}  // namespace fg
