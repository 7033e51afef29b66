/*
 * fg.h -- C ABI of libfg.so: the OPT-style transformer layer of FlexGen on
 * weights and KV cache stored in fine-grained asymmetric 4-bit groups of 64,
 * for one NVIDIA GB300 (sm_103a).
 *
 * Sources (FlexGen notes, papercache.org, "FlexGen: High-Throughput Generative
 * Inference of Large Language Models with a Single GPU"):
 *   [BG]  section "背景知识" (Background): the prefill equations
 *         x_K = x w_K, x_V = x w_V, x_Q = x w_Q,
 *         x_Out = Softmax(x_Q x_K^T / sqrt(h1)) x_V w_O + x,
 *         x' = relu(x_Out w_1) w_2 + x_Out,
 *         and the decode equations with KV Concat for t in R^{b x 1 x h1}.
 *   [S5]  section "5. 近似方法" (Approximate Methods): group-wise asymmetric
 *         quantization x_q = round((x - min)/(max - min) * (2^b - 1)), b = 4,
 *         g = 64, weights grouped along the output channel, KV along the
 *         hidden dimension, stored quantized and converted back to FP16
 *         before compute.
 *   [S4]  section "4. 卸载策略": the zig-zag block schedule -- one load of a
 *         layer's weights serves every sequence of the block.
 *
 * Conventions for every entry point:
 *   - All pointers named "device" are CUDA device pointers on the current
 *     device; the caller owns every buffer.  The library never allocates
 *     device memory and keeps no per-call state on the host.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream).
 *     Argument errors are returned synchronously before anything is
 *     launched; a failed launch returns FG_ERR_CUDA.  Errors raised inside a
 *     kernel (a bounded wait that ran out) are reported by fg_sync_status.
 *   - Grouping is always along the innermost, contiguous dimension of the
 *     tensor named, in groups of 64 consecutive elements.  A 4-bit tensor
 *     of logical shape [R][C] is three arrays:
 *         codes  uint8 [R][C/2]   byte j = q[2j] | q[2j+1] << 4
 *         mins   fp32  [R][C/64]  group minimum
 *         scales fp32  [R][C/64]  (max - min) / 15
 *     and element (r, c) is restored as fmaf(q, scale, min) in fp32
 *     (then rounded to fp16 when the consumer computes in fp16).
 *   - Codes and activations must be 16-byte aligned (FG_ERR_ALIGN), mins and
 *     scales 4-byte aligned.
 *   - No CPU fallback exists: every operation runs in the library's CUDA
 *     kernels.
 */
#ifndef FG_H_
#define FG_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FG_OK = 0,
  FG_ERR_ARG = 1,             /* null pointer, negative size, bad enum      */
  FG_ERR_SHAPE = 2,           /* a dimension breaks a divisibility rule     */
  FG_ERR_ALIGN = 3,           /* pointer alignment                          */
  FG_ERR_CAPACITY = 4,        /* KV slot outside [0, capacity)              */
  FG_ERR_WORKSPACE = 5,       /* workspace null or smaller than required   */
  FG_ERR_CUDA = 6,            /* a CUDA runtime call or launch failed       */
  FG_ERR_DEVICE_TIMEOUT = 7,  /* a kernel gave up a bounded wait            */
  FG_ERR_UNSUPPORTED = 8      /* valid, but not implemented (e.g. head_dim) */
} fg_status;

typedef enum { FG_F16 = 0, FG_F32 = 1 } fg_dtype;               /* activations */
typedef enum { FG_CODEC_NONE = 0, FG_CODEC_Q4G64 = 1 } fg_codec; /* storage     */

/* One weight matrix w in R^{K x N}, used as x . w ([BG]); K = input
 * features, N = output features.  With FG_CODEC_Q4G64: codes [K][N/2],
 * mins and scales [K][N/64] -- each group is 64 consecutive output channels
 * at one input index ([S5]: "along the output-channel dimension").  With
 * FG_CODEC_NONE: dense [K][N] in the layer's activation dtype.  Device.
 * packed (optional, may be NULL): the decode copy written by fg_pack_weight
 * in format packed_format (an fg_pack_format); fp16 products of up to 256
 * rows read it instead of codes/mins/scales. */
typedef struct {
  const uint8_t* codes;
  const float* mins;
  const float* scales;
  const void* dense;
  int64_t K, N;
  const uint8_t* packed;
  int32_t packed_format;
} fg_wmat;

/* Formats of the decode copy of a Q4G64 weight (fg_pack_weight).
 *   FG_PACK_EXACT (default): the stored fp32 (min, scale) of every group, so
 *     a decode product restores each weight as fp16(fmaf(q, scale, min)),
 *     exactly the value fg_dequant_g64 writes ([S5] "converted back to FP16
 *     before compute"); 0.625 bytes per weight, like the stored form.
 *   FG_PACK_F16META (opt-in, approximate): (scale, min) rounded to fp16 and
 *     applied in fp16, w~ = fp16(q * fp16(scale) + fp16(min)) with one
 *     rounding; 0.5625 bytes per weight (10% fewer bytes to read).  Bound:
 *     |w~ - x| <= scale/2 + 15 * ulp16(scale)/2 + ulp16(min)/2 + ulp16(w~)/2
 *     + the fp32 codec's own rounding, for finite groups whose scale and
 *     min are normal fp16 numbers. */
typedef enum { FG_PACK_EXACT = 0, FG_PACK_F16META = 1 } fg_pack_format;

/* One transformer layer ([BG]): w_Q, w_K, w_V, w_O in R^{h1 x h1},
 * w_1 in R^{h1 x h2}, w_2 in R^{h2 x h1}; `heads` attention heads of
 * head_dim = h1 / heads (score scale 1/sqrt(head_dim); heads = 1 is the
 * page's 1/sqrt(h1)).  h1 and h2 must be multiples of 64; head_dim must be
 * 64 or 128. */
typedef struct {
  fg_wmat wq, wk, wv, wo, w1, w2;
  int64_t h1, h2;
  int32_t heads;
  fg_codec codec;
  fg_dtype dtype;
} fg_layer;

/* One layer's KV cache for b sequences ([BG] x_K, x_V, grown by Concat).
 * Layout [b][heads][capacity][head_dim]; a token's K (or V) row of h1 =
 * heads * head_dim values is quantized in groups of 64 along the hidden
 * dimension ([S5]), which never straddle heads because head_dim % 64 == 0.
 *   FG_CODEC_Q4G64: {k,v}_codes uint8 [b][H][cap][d/2],
 *                   {k,v}_mins, {k,v}_scales fp32 [b][H][cap][d/64]
 *   FG_CODEC_NONE:  {k,v}_dense [b][H][cap][d] in `dtype`.
 * Device memory owned by the caller; slot p holds the token at position p. */
typedef struct {
  uint8_t* k_codes;
  uint8_t* v_codes;
  float* k_mins;
  float* k_scales;
  float* v_mins;
  float* v_scales;
  void* k_dense;
  void* v_dense;
  int64_t b, capacity;
  int32_t heads, head_dim;
  fg_codec codec;
  fg_dtype dtype;
} fg_kv;

/* [S5] quantization equation.  x: device [rows][cols] of dtype `dt`
 * (fp16 or fp32), cols % 64 == 0.  Writes codes [rows][cols/2], mins and
 * scales [rows][cols/64].  Per group, in IEEE fp32 with round-to-nearest-
 * even and no contraction: min/max in the total order of non-NaN values
 * (-0 < +0; an all-NaN group gives NaN), r = max - min, scale = r / 15,
 * q = clamp(rint(((x - min) / r) * 15), 0, 15) with a NaN quotient -> 0.
 * rows == 0 is a no-op. */
fg_status fg_quantize_g64(const void* x, fg_dtype dt, int64_t rows, int64_t cols,
                          uint8_t* codes, float* mins, float* scales, cudaStream_t stream);

/* [S5] "converted back to FP16 before compute".  Inverse of the layout
 * above: out[r][c] = fmaf(q, scale, min) in fp32, stored as `dt` (fp16:
 * round-to-nearest-even).  out: device [rows][cols]. */
fg_status fg_dequant_g64(const uint8_t* codes, const float* mins, const float* scales,
                         int64_t rows, int64_t cols, void* out, fg_dtype dt,
                         cudaStream_t stream);

/* [BG] decode, "x_K <- Concat(x_K, t w_K); x_V <- Concat(x_V, t w_V)":
 * store the rows k_new, v_new (device [kv->b][h1], kv->dtype) at slot `pos`
 * of every sequence, quantizing each 64-group of the hidden dimension with
 * the fg_quantize_g64 arithmetic when kv->codec is FG_CODEC_Q4G64.
 * pos outside [0, capacity) -> FG_ERR_CAPACITY. */
fg_status fg_kv_append(const fg_kv* kv, const void* k_new, const void* v_new, int64_t pos,
                       cudaStream_t stream);

/* [BG] one product of the layer with its epilogue, on weights stored per
 * [S5]: y = act(x . w + r), act = relu if `relu` != 0 else identity.
 * x: device [M][w->K] (dtype), r: device [M][w->N] or NULL, y: device
 * [M][w->N]; y must not overlap x or r.
 * codec FG_CODEC_Q4G64 uses w->codes/mins/scales (dequantized on the fly,
 * rounded to the compute dtype), FG_CODEC_NONE uses w->dense ([K][N] in
 * dtype).  K and N must be multiples of 64.  fp16 on Q4G64 weights with a
 * decode copy (w->packed): M <= 256 runs on the tensor cores (weights
 * converted into tensor memory); without the copy, M >= 64 runs on the
 * tensor cores after converting the weight to fp16 in ws.  fp16 dense
 * weights with M >= 64 run on the tensor cores; other cases on the CUDA
 * cores.  Products are split over K when the output has too few tiles,
 * using ws.  ws_bytes >= fg_linear_workspace_bytes. */
size_t fg_linear_workspace_bytes(int64_t M, int64_t K, int64_t N, fg_codec codec, fg_dtype dtype);
fg_status fg_linear(const fg_wmat* w, fg_codec codec, fg_dtype dtype, const void* x, int64_t M,
                    const void* r, int32_t relu, void* y, void* ws, size_t ws_bytes,
                    cudaStream_t stream);

/* The decode copy of a Q4G64 weight ([S5] storage; [BG] x . w with one
 * weight read for the whole block) in `format` (fg_pack_format):
 * fg_pack_weight_bytes(K, N, format) = (K/64) * (N/128) blocks of B bytes,
 * B = 5120 (FG_PACK_EXACT) or 4608 (FG_PACK_F16META): one block per
 * (128-channel tile t, 64-k tile u), block (t, u) at byte offset
 * (t * K/64 + u) * B, so the k tiles of a channel tile are one contiguous run:
 *   bytes 0..4095: codes, 16-byte units [q][g2][t] (q = 0..3, g2 = 0..1,
 *     t = 0..31) at q*1024 + g2*512 + t*16; 32-bit word w of unit (q, g2, t)
 *     holds channel 32q + t/4 + 8w of the tile at the tile's k pairs
 *     j = 16*g2 + 4e + t%4, e = 0..3: nibble e (from the low end) is k = 2j,
 *     nibble e+4 is k = 2j+1, so one mask turns a word into fp16 pairs of
 *     consecutive k;
 *   FG_PACK_EXACT, bytes 4096..5119: for the tile's two 64-channel groups gl
 *     (lower first) and its k pairs j = 0..31, the 16-byte unit at
 *     4096 + gl*512 + j*16 holds fp32 (scale[2j], scale[2j+1], min[2j],
 *     min[2j+1]) as stored;
 *   FG_PACK_F16META, bytes 4096..4607: for the groups gl, 16-byte units at
 *     4096 + gl*256 + (u*4 + c)*16, u = 0..3, c = 0..3: fp16x2 (scale[2j],
 *     scale[2j+1]), fp16x2 (min[2j], min[2j+1]) for j = 8u + c, then the same
 *     for j = 8u + 4 + c; each rounded to nearest even.
 *   (The order is the one in which the converting threads read them: thread
 *   t of warp quarter q converts channels 32q + t/4 + 8w at the k pairs
 *   4i + t%4, the register order of a 16x128b tensor-memory store.)
 * packed: device, 16-byte aligned, owned by the caller, then stored in
 * w->packed with w->packed_format = format.  K a multiple of 64 and N of
 * 128, else FG_ERR_SHAPE; null arrays or an unknown format -> FG_ERR_ARG
 * (fg_pack_weight_bytes returns 0 for those).  Asynchronous on `stream`. */
size_t fg_pack_weight_bytes(int64_t K, int64_t N, int32_t format);
fg_status fg_pack_weight(const fg_wmat* w, int32_t format, uint8_t* packed, cudaStream_t stream);

/* [BG] decode attention alone: for every sequence and head,
 * Softmax(q K^T / sqrt(head_dim)) V over cache slots 0..pos of kv (nothing
 * is appended), K/V read through the codec.  q: device [kv->b][ldq] with
 * head h at columns h*head_dim (dtype kv->dtype); out: device [kv->b][ldo],
 * same layout.  ldq and ldo are multiples of 8 and at least h1.  The cache
 * is split over tokens when there are too few (sequence, head) pairs to fill
 * the GPU; the split partials use ws (device, ws_bytes >=
 * fg_decode_attention_workspace_bytes(kv), 0 when no split is needed).
 * pos outside [0, capacity) -> FG_ERR_CAPACITY. */
size_t fg_decode_attention_workspace_bytes(const fg_kv* kv);
fg_status fg_decode_attention(const fg_kv* kv, const void* q, int64_t ldq, int64_t pos, void* out,
                              int64_t ldo, void* ws, size_t ws_bytes, cudaStream_t stream);

/* [S5] sparse attention ("4-bit-S"): decode attention that keeps, for each
 * sequence and head, only the `keep` tokens of slots 0..pos with the largest
 * scores q.k/sqrt(head_dim) and reads only their rows of V:
 *   out = sum over the kept i of p_i v_i,  p = Softmax(q K^T / sqrt(d))
 * over ALL pos+1 tokens (the kept weights are not renormalised).  Among equal
 * scores the lower slot ranks first.  keep >= pos+1 keeps every token (dense
 * attention); the page's setting keeps the top 10%, ceil((pos+1)/10).
 * q, out, ldq, ldo as for fg_decode_attention; nothing is appended.
 * idx: optional device int32 [kv->b][heads][min(keep, pos+1)], 4-byte
 * aligned, receives the kept slots of each (sequence, head) in ascending
 * order; NULL to skip.  Needs a 4-bit cache with fp16 activations and
 * pos+1 <= 16384 (else FG_ERR_UNSUPPORTED); keep < 1 -> FG_ERR_ARG; pos
 * outside [0, capacity) -> FG_ERR_CAPACITY.  No workspace.  Asynchronous on
 * `stream`.  A cache holding NaN gives NaN outputs; which slots are then
 * reported is unspecified. */
fg_status fg_decode_attention_topk(const fg_kv* kv, const void* q, int64_t ldq, int64_t pos, int64_t keep,
                                   void* out, int64_t ldo, int32_t* idx, cudaStream_t stream);

/* fg_decode_attention for callers that cannot allocate device memory: code
 * embedded in a host application that owns the GPU memory pool and forbids
 * other allocations, or a latency-critical loop that cannot afford the
 * device-wide synchronization a cudaMalloc/cudaFree may imply.  (The FlexGen
 * notes have no counterpart; this is an interface convenience.)
 * Same arguments and results as fg_decode_attention, without a workspace:
 * the split partials go to a 1 MiB array built into libfg.so, which every
 * GPU that loads the library holds until the process exits.  Caches whose
 * fg_decode_attention_workspace_bytes exceeds 1 MiB are rejected with
 * FG_ERR_WORKSPACE (the split rule needs at most ~0.9 MB, so none is
 * today).  Argument errors are reported before any CUDA call, as for
 * fg_decode_attention.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress, with that device current) and caches
 * it until the process exits; make that first call before any stream
 * capture and before any region where allocations are forbidden (under lazy
 * module loading it is also the call that loads this code, and the array,
 * onto the device).  After a device reset (or a destroyed primary context)
 * the cached address is stale: do not call this entry point again in that
 * process.  Calls share the array, so calls whose kernels overlap on the GPU
 * (concurrent streams) race; nothing in the array needs to start at zero.
 * Calls no allocating routine, on the device or the host (the array is part
 * of the library's device code; under lazy module loading the driver places
 * it on the device when the first call loads that code). */
fg_status fg_decode_attention_noalloc(const fg_kv* kv, const void* q, int64_t ldq, int64_t pos,
                                      void* out, int64_t ldo, cudaStream_t stream);

/* Workspace (device bytes) that fg_prefill_layer / fg_prefill_block need for
 * b sequences of s tokens, and that fg_decode_step / fg_decode_block_step
 * need for b sequences with a cache of `capacity` slots.  Pure host
 * functions; 0 on invalid arguments. */
size_t fg_prefill_workspace_bytes(const fg_layer* L, int64_t b, int64_t s);
size_t fg_decode_workspace_bytes(const fg_layer* L, int64_t b, int64_t capacity);

/* [BG] prefill of one layer.  x: device [b][s][h1] (L->dtype); y: device
 * [b][s][h1] output x^{i+1}, must not overlap x.  Writes K/V rows of the s
 * prompt tokens into slots 0..s-1 of kv (quantized per [S5]); attention is
 * causal and reads K/V back through the codec, so the new tokens see the
 * same values a later decode step reads.  Requires kv->b == b,
 * s <= kv->capacity, and ws_bytes >= fg_prefill_workspace_bytes(L, b, s).
 * fp16 layers with a 4-bit cache, s a multiple of 128 and head_dim 64 or
 * 128 run the attention on the tensor cores (tcgen05), one CTA per SM;
 * other prompts take the warp-level MMA kernel.  Both give the same values
 * up to rounding. */
fg_status fg_prefill_layer(const fg_layer* L, const void* x, int64_t b, int64_t s,
                           const fg_kv* kv, void* y, void* ws, size_t ws_bytes,
                           cudaStream_t stream);

/* [BG] one decode step of one layer for the whole block (zig-zag reuse [S4]:
 * each weight is read once for all b sequences).  t: device [b][h1]; appends
 * t w_K, t w_V at slot `pos` (Concat), attends over slots 0..pos and writes
 * t^{i+1} to y (device [b][h1], must not overlap t).  pos outside
 * [0, capacity) -> FG_ERR_CAPACITY. */
fg_status fg_decode_step(const fg_layer* L, const void* t, int64_t b, int64_t pos,
                         const fg_kv* kv, void* y, void* ws, size_t ws_bytes,
                         cudaStream_t stream);

/* [S4] zig-zag block, prefill half: run the prompt x (device [b][s][h1])
 * through layers[0..l-1] with caches kvs[0..l-1]; the last layer's output
 * goes to y (device [b][s][h1]).  Workspace as for fg_prefill_layer plus
 * 2*b*s*h1 activation elements (see fg_prefill_block_workspace_bytes). */
size_t fg_prefill_block_workspace_bytes(const fg_layer* L, int64_t b, int64_t s);
fg_status fg_prefill_block(const fg_layer* layers, int32_t l, const void* x, int64_t b,
                           int64_t s, const fg_kv* kvs, void* y, void* ws, size_t ws_bytes,
                           cudaStream_t stream);

/* [S4] zig-zag block, one generation step: feed t (device [b][h1]) through
 * every layer at slot `pos`; the last layer's output goes to y. */
size_t fg_decode_block_workspace_bytes(const fg_layer* L, int64_t b, int64_t capacity);
fg_status fg_decode_block_step(const fg_layer* layers, int32_t l, const void* t, int64_t b,
                               int64_t pos, const fg_kv* kvs, void* y, void* ws,
                               size_t ws_bytes, cudaStream_t stream);

/* [S4] Algorithm 1 on GB300: the zig-zag block's decode step with the
 * weights offloaded to host memory (the Grace LPDDR behind NVLink-C2C).
 * layers[] are fp16 4-bit layers whose decode copies (w->packed, all six
 * matrices, one format) may live in host memory (pinned, or any memory
 * cudaMemcpyAsync reads); the decode kernels read nothing else of a weight.
 * Layer by layer, the six copies are copied on `copy_stream` into one of
 * two halves of `stage` (device, 256-byte aligned, stage_bytes >=
 * fg_offload_stage_bytes(&layers[0])) while `stream` computes the previous
 * layer from the other half: the load of layer i+1 overlaps the compute of
 * layer i.  Events order the halves between the two streams (a per-device
 * set kept by the library: calls on one device must not overlap).  Same
 * arguments, results and errors as fg_decode_block_step otherwise; the
 * outputs are bit-identical to it.  copy_stream may equal stream (no
 * overlap).  Layers that need no decode copy -> FG_ERR_UNSUPPORTED. */
size_t fg_offload_stage_bytes(const fg_layer* L);
fg_status fg_decode_block_step_offload(const fg_layer* layers, int32_t l, const void* t, int64_t b, int64_t pos,
                                       const fg_kv* kvs, void* y, void* ws, size_t ws_bytes, void* stage,
                                       size_t stage_bytes, cudaStream_t stream, cudaStream_t copy_stream);

/* [S4] the zig-zag block's decode step replayed as a CUDA graph: the same
 * arguments, results and errors as fg_decode_block_step.  The first call
 * with a given set of arguments (every pointer and size, and the bytes of
 * the layers[] and kvs[] structures) runs the step directly and then
 * records its launches into a graph held by `cache`; later calls with the
 * same arguments launch that graph, one host call per step.  Buffers the
 * graphs refer to must stay allocated while `cache` holds them.  While
 * fg_profile_start is active, or when `stream` is itself being captured,
 * calls run the step directly and record nothing.  A cache may be shared by
 * host threads; graphs launch on the stream each call names (recording uses
 * a stream of the cache's own, on the current device: one device per
 * cache). */
typedef struct fg_graph_cache fg_graph_cache;
fg_status fg_graph_cache_create(fg_graph_cache** cache);
void fg_graph_cache_destroy(fg_graph_cache* cache);
int64_t fg_graph_cache_size(const fg_graph_cache* cache);   /* graphs held */
fg_status fg_decode_block_step_graphed(fg_graph_cache* cache, const fg_layer* layers, int32_t l, const void* t,
                                       int64_t b, int64_t pos, const fg_kv* kvs, void* y, void* ws,
                                       size_t ws_bytes, cudaStream_t stream);

/* Synchronize `stream`, then report (and clear) the device error word that
 * kernels raise when a bounded wait runs out: FG_ERR_DEVICE_TIMEOUT, or
 * FG_ERR_CUDA if the synchronization itself failed. */
#define FG_WAIT_LIMIT_DEFAULT (1u << 24)

/* Failure handling: the number of polls every bounded wait of the library's
 * kernels makes (on copies landing, on other warps' stages) before it gives
 * up, sets the device error word and lets its CTA leave -- after the CTA's
 * own copies and tensor-core operations in flight have completed and its
 * tensor memory is freed -- so that a lost dependency ends in
 * FG_ERR_DEVICE_TIMEOUT from fg_sync_status instead of a hang.  Process-wide,
 * read at each launch; 0 makes every such wait give up at once (outputs are
 * then undefined).  Returns the previous value; FG_WAIT_LIMIT_DEFAULT is the
 * initial one. */
uint32_t fg_set_wait_limit(uint32_t polls);
fg_status fg_sync_status(cudaStream_t stream);

/* Human-readable name of a status, and the detail message of the most recent
 * failing call on this host thread ("" if none). */
const char* fg_status_str(fg_status s);
const char* fg_last_error(void);

/* Launch accounting (measurement support, not part of the method).
 * fg_profile_start(max_launches): from now on the library's kernel launches
 * are timed with CUDA events on their own stream (host-side event objects,
 * no device memory).  Launches of one class that follow one another on a
 * stream form one run with one event pair, so that consecutive products
 * keep their programmatic overlap; up to max_launches runs, later ones are
 * counted as dropped.  fg_profile_stop(): waits for the recorded events and
 * accumulates launches and time per (phase, kernel class)
 * (FG_ERR_WORKSPACE if runs were dropped).  fg_profile_phase(p), 0 <= p < 4: tags the following
 * launches with phase p (0 after start), e.g. prefill vs decode.
 * fg_profile_query(p, i, ...): launches and total milliseconds of class i
 * (0 <= i < fg_profile_kernel_classes()) in phase p, named by
 * fg_profile_kernel_name(i).  Not thread-safe against concurrent
 * start/stop.  fg_launch_count(): kernels launched since the library
 * was loaded. */
fg_status fg_profile_start(int32_t max_launches);
fg_status fg_profile_phase(int32_t phase);
fg_status fg_profile_stop(void);
int32_t fg_profile_kernel_classes(void);
const char* fg_profile_kernel_name(int32_t i);
fg_status fg_profile_query(int32_t phase, int32_t i, int64_t* launches, double* total_ms);
uint64_t fg_launch_count(void);

/* Library version, e.g. "fg 0.1 sm_103a". */
const char* fg_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FG_H_ */
