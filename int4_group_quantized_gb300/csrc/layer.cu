// The OPT-style layer and the zig-zag block loop (FlexGen notes, "背景知识"
// prefill and decode equations; "4. 卸载策略" zig-zag block schedule with the
// whole block resident, so one pass over a layer's weights serves every
// sequence of the block).  Argument validation, workspace layout and the
// sequence of kernel launches live here; the arithmetic is in the kernels.
#include <mutex>

#include "fg_internal.cuh"

namespace fg {
namespace {

constexpr size_t kAlign = 256;
inline size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

fg_status check_wmat(const fg_wmat& w, int64_t K, int64_t N, fg_codec codec, const char* name) {
  if (w.K != K || w.N != N)
    return fail(FG_ERR_SHAPE, "%s is %lldx%lld, expected %lldx%lld", name, (long long)w.K,
                (long long)w.N, (long long)K, (long long)N);
  if (codec == FG_CODEC_Q4G64) {
    if (!w.codes || !w.mins || !w.scales) return fail(FG_ERR_ARG, "%s: null 4-bit arrays", name);
    if (!aligned(w.codes, 16) || !aligned(w.mins, 4) || !aligned(w.scales, 4))
      return fail(FG_ERR_ALIGN, "%s: codes need 16-byte alignment", name);
    if (w.packed && !aligned(w.packed, 16)) return fail(FG_ERR_ALIGN, "%s: packed copy needs 16-byte alignment", name);
    if (w.packed && w.packed_format != FG_PACK_EXACT && w.packed_format != FG_PACK_F16META)
      return fail(FG_ERR_ARG, "%s: unknown packed_format %d", name, w.packed_format);
  } else {
    if (!w.dense) return fail(FG_ERR_ARG, "%s: null dense weights", name);
    if (!aligned(w.dense, 16)) return fail(FG_ERR_ALIGN, "%s: dense weights need 16-byte alignment", name);
  }
  return FG_OK;
}

fg_status check_layer(const fg_layer* L) {
  if (!L) return fail(FG_ERR_ARG, "null layer");
  if (L->dtype != FG_F16 && L->dtype != FG_F32) return fail(FG_ERR_ARG, "layer dtype");
  if (L->codec != FG_CODEC_NONE && L->codec != FG_CODEC_Q4G64) return fail(FG_ERR_ARG, "layer codec");
  if (L->h1 <= 0 || L->h2 <= 0 || L->heads <= 0) return fail(FG_ERR_ARG, "layer sizes");
  if (L->h1 % 64 || L->h2 % 64) return fail(FG_ERR_SHAPE, "h1 and h2 must be multiples of 64");
  if (L->h1 % L->heads) return fail(FG_ERR_SHAPE, "heads must divide h1");
  const int64_t d = L->h1 / L->heads;
  if (d != 64 && d != 128) return fail(FG_ERR_UNSUPPORTED, "head_dim %lld (64 or 128)", (long long)d);
  fg_status s;
  const int64_t h1 = L->h1, h2 = L->h2;
  if ((s = check_wmat(L->wq, h1, h1, L->codec, "w_Q")) != FG_OK) return s;
  if ((s = check_wmat(L->wk, h1, h1, L->codec, "w_K")) != FG_OK) return s;
  if ((s = check_wmat(L->wv, h1, h1, L->codec, "w_V")) != FG_OK) return s;
  if ((s = check_wmat(L->wo, h1, h1, L->codec, "w_O")) != FG_OK) return s;
  if ((s = check_wmat(L->w1, h1, h2, L->codec, "w_1")) != FG_OK) return s;
  if ((s = check_wmat(L->w2, h2, h1, L->codec, "w_2")) != FG_OK) return s;
  return FG_OK;
}

fg_status check_kv(const fg_kv* kv, int64_t b, int32_t heads, int64_t d, fg_codec codec,
                   fg_dtype dt) {
  if (!kv) return fail(FG_ERR_ARG, "null kv");
  if (kv->codec != codec || kv->dtype != dt) return fail(FG_ERR_ARG, "kv codec/dtype differ from the layer");
  if (kv->heads != heads || kv->head_dim != d)
    return fail(FG_ERR_SHAPE, "kv heads/head_dim %d/%d, layer %d/%lld", kv->heads, kv->head_dim,
                heads, (long long)d);
  if (kv->b != b) return fail(FG_ERR_SHAPE, "kv holds %lld sequences, call has %lld", (long long)kv->b, (long long)b);
  if (kv->capacity <= 0) return fail(FG_ERR_ARG, "kv capacity");
  if (codec == FG_CODEC_Q4G64) {
    if (!kv->k_codes || !kv->v_codes || !kv->k_mins || !kv->k_scales || !kv->v_mins || !kv->v_scales)
      return fail(FG_ERR_ARG, "kv: null 4-bit arrays");
    if (!aligned(kv->k_codes, 16) || !aligned(kv->v_codes, 16) || !aligned(kv->k_mins, 4) ||
        !aligned(kv->k_scales, 4) || !aligned(kv->v_mins, 4) || !aligned(kv->v_scales, 4))
      return fail(FG_ERR_ALIGN, "kv: codes need 16-byte alignment");
  } else {
    if (!kv->k_dense || !kv->v_dense) return fail(FG_ERR_ARG, "kv: null dense arrays");
    if (!aligned(kv->k_dense, 16) || !aligned(kv->v_dense, 16)) return fail(FG_ERR_ALIGN, "kv: dense arrays need 16-byte alignment");
  }
  return FG_OK;
}

WSeg seg_of(const fg_wmat& w, int64_t n0) {
  WSeg s;
  s.codes = w.codes;
  s.packed = w.packed;
  s.packed_format = w.packed_format;
  s.mins = w.mins;
  s.scales = w.scales;
  s.dense = w.dense;
  s.N = w.N;
  s.n0 = n0;
  return s;
}

GemmArgs product(const fg_layer& L, const void* X, int64_t ldx, int64_t M, const fg_wmat* ws,
                 int nseg, void* Y, int64_t ldy, const void* R, int64_t ldr, int relu) {
  GemmArgs a{};
  a.X = X;
  a.ldx = ldx;
  a.M = M;
  a.K = ws[0].K;
  int64_t n0 = 0;
  for (int i = 0; i < nseg; ++i) {
    a.seg[i] = seg_of(ws[i], n0);
    n0 += ws[i].N;
  }
  a.nseg = nseg;
  a.N = n0;
  a.Y = Y;
  a.ldy = ldy;
  a.R = R;
  a.ldr = ldr;
  a.relu = relu;
  a.quant = L.codec == FG_CODEC_Q4G64;
  a.dtype = L.dtype;
  return a;
}

// Workspace carve-up shared by prefill (M = b*s) and decode (M = b).
struct Buffers {
  char* qkv;  // [M][3 h1]
  char* att;  // [M][h1]
  char* xo;   // [M][h1]
  char* hid;  // [M][h2]
  char* scratch;
  size_t scratch_bytes;
};

size_t activations_bytes(const fg_layer& L, int64_t M) {
  const size_t e = dtype_bytes(L.dtype);
  return up(M * 3 * L.h1 * e) + up(M * L.h1 * e) * 2 + up(M * L.h2 * e);
}

// Prefill with fp16 activations runs its products from fp16 weights: the
// layer's six 4-bit matrices are dequantized once into the workspace (each
// weight then feeds all b*s rows).
bool prefill_dequantizes(const fg_layer& L, int64_t) {
  return L.dtype == FG_F16 && L.codec == FG_CODEC_Q4G64;
}

// fp16 decode products on 4-bit weights read the decode copy of every
// matrix (fg_pack_weight): one launch per product, the weights converted in
// registers.  A layer without it is rejected rather than run on a slower path.
bool decode_needs_copies(const fg_layer& L) { return L.dtype == FG_F16 && L.codec == FG_CODEC_Q4G64; }

fg_status check_decode_copies(const fg_layer& L) {
  if (!decode_needs_copies(L)) return FG_OK;
  const fg_wmat* m[6] = {&L.wq, &L.wk, &L.wv, &L.wo, &L.w1, &L.w2};
  const char* names[6] = {"w_Q", "w_K", "w_V", "w_O", "w_1", "w_2"};
  for (int i = 0; i < 6; ++i) {
    if (!m[i]->packed)
      return fail(FG_ERR_ARG, "%s has no decode copy: fp16 decode needs fg_pack_weight on every matrix", names[i]);
    if (m[i]->packed_format != L.wq.packed_format)
      return fail(FG_ERR_ARG, "%s: the decode copies of a layer must share one format", names[i]);
  }
  if (L.h1 % 128 || L.h2 % 128) return fail(FG_ERR_SHAPE, "fp16 decode needs h1 and h2 multiples of 128");
  return FG_OK;
}
size_t w16_bytes(const fg_layer& L) {
  return up(L.h1 * L.h1 * 2) * 4 + up(L.h1 * L.h2 * 2) * 2;
}

size_t scratch_bytes(const fg_layer& L, int64_t M, int64_t capacity, bool decode) {
  int quant = L.codec == FG_CODEC_Q4G64;
  const bool packed = decode && decode_needs_copies(L);
  size_t w16 = 0;
  if (!decode && prefill_dequantizes(L, M)) {
    w16 = w16_bytes(L);
    quant = 0;
  }
  size_t s = gemm_workspace_bytes(M, 3 * L.h1, L.h1, L.dtype, quant, packed);
  size_t t = gemm_workspace_bytes(M, L.h1, L.h1, L.dtype, quant, packed);
  s = t > s ? t : s;
  t = gemm_workspace_bytes(M, L.h2, L.h1, L.dtype, quant, packed);
  s = t > s ? t : s;
  t = gemm_workspace_bytes(M, L.h1, L.h2, L.dtype, quant, packed);
  s = t > s ? t : s;
  if (decode) {
    t = decode_attention_workspace_bytes(M, L.heads, static_cast<int32_t>(L.h1 / L.heads), capacity);
    s = t > s ? t : s;
  }
  return w16 + up(s);
}

Buffers carve(const fg_layer& L, int64_t M, void* ws) {
  const size_t e = dtype_bytes(L.dtype);
  Buffers B;
  char* p = static_cast<char*>(ws);
  B.qkv = p;
  p += up(M * 3 * L.h1 * e);
  B.att = p;
  p += up(M * L.h1 * e);
  B.xo = p;
  p += up(M * L.h1 * e);
  B.hid = p;
  p += up(M * L.h2 * e);
  B.scratch = p;
  return B;
}

fg_status run_prefill(const fg_layer& L, const void* x, int64_t b, int64_t s, const fg_kv& kv,
                      void* y, void* ws, size_t scratch, cudaStream_t st) {
  const int64_t M = b * s, h1 = L.h1, h2 = L.h2;
  Buffers B = carve(L, M, ws);
  fg_layer Lc = L;   // the layer as the products see it
  if (prefill_dequantizes(L, M)) {
    // "converted back to FP16 before compute": once per layer, into the workspace
    char* w = B.scratch;
    fg_wmat* mats[6] = {&Lc.wq, &Lc.wk, &Lc.wv, &Lc.wo, &Lc.w1, &Lc.w2};
    for (fg_wmat* m : mats) {
      FG_TRY(dequant_rows(m->codes, m->mins, m->scales, m->K, m->N, w, FG_F16, st));
      m->dense = w;
      m->codes = nullptr;
      w += up(m->K * m->N * 2);
    }
    Lc.codec = FG_CODEC_NONE;
    scratch -= w16_bytes(L);
    B.scratch = w;
  }
  const fg_layer& P = Lc;
  const fg_wmat qkv[3] = {P.wq, P.wk, P.wv};
  // x_Q, x_K, x_V = x w_Q, x w_K, x w_V (one pass over the three matrices)
  FG_TRY(gemm(product(P, x, h1, M, qkv, 3, B.qkv, 3 * h1, nullptr, 0, 0), B.scratch, scratch, st));
  // cache the prompt's K/V (quantized per token along the hidden dimension);
  // on the tensor-core attention path the K/V columns then hold what the
  // cache restores
  const size_t e = dtype_bytes(L.dtype);
  const int32_t d = static_cast<int32_t>(h1 / L.heads);
  const bool tc = kv.codec == FG_CODEC_Q4G64 && prefill_attention_tc_supported(s, d, L.dtype);
  FG_TRY(kv_store(kv, B.qkv + h1 * e, B.qkv + 2 * h1 * e, 3 * h1, b, s, 0, st, tc));
  // Softmax(x_Q x_K^T / sqrt(d)) x_V, causal, K/V read back through the codec
  if (tc)
    FG_TRY(prefill_attention_tc(B.qkv, 3 * h1, b, s, L.heads, d, B.att, h1, st));
  else
    FG_TRY(prefill_attention(kv, B.qkv, 3 * h1, b, s, B.att, h1, st));
  // x_Out = (...) w_O + x
  FG_TRY(gemm(product(P, B.att, h1, M, &P.wo, 1, B.xo, h1, x, h1, 0), B.scratch, scratch, st));
  // relu(x_Out w_1)
  FG_TRY(gemm(product(P, B.xo, h1, M, &P.w1, 1, B.hid, h2, nullptr, 0, 1), B.scratch, scratch, st));
  // x^{i+1} = (...) w_2 + x_Out
  FG_TRY(gemm(product(P, B.hid, h2, M, &P.w2, 1, y, h1, B.xo, h1, 0), B.scratch, scratch, st));
  return FG_OK;
}

fg_status run_decode(const fg_layer& L, const void* t, int64_t b, int64_t pos, const fg_kv& kv,
                     void* y, void* ws, size_t scratch, cudaStream_t st) {
  const int64_t h1 = L.h1, h2 = L.h2;
  Buffers B = carve(L, b, ws);
  const fg_wmat qkv[3] = {L.wq, L.wk, L.wv};
  // t_Q, t w_K, t w_V: every weight read once for the whole block
  FG_TRY(gemm(product(L, t, h1, b, qkv, 3, B.qkv, 3 * h1, nullptr, 0, 0), B.scratch, scratch, st));
  // Concat (t w_K, t w_V into slot pos), then Softmax(t_Q x_K^T / sqrt(d)) x_V
  // over slots 0..pos
  const size_t e = dtype_bytes(L.dtype);
  FG_TRY(decode_attention(kv, B.qkv, 3 * h1, B.qkv + h1 * e, B.qkv + 2 * h1 * e, 3 * h1, b, pos,
                          B.att, h1, B.scratch, scratch, st));
  FG_TRY(gemm(product(L, B.att, h1, b, &L.wo, 1, B.xo, h1, t, h1, 0), B.scratch, scratch, st));
  FG_TRY(gemm(product(L, B.xo, h1, b, &L.w1, 1, B.hid, h2, nullptr, 0, 1), B.scratch, scratch, st));
  FG_TRY(gemm(product(L, B.hid, h2, b, &L.w2, 1, y, h1, B.xo, h1, 0), B.scratch, scratch, st));
  return FG_OK;
}

fg_status check_act(const void* p, const char* name) {
  if (!p) return fail(FG_ERR_ARG, "%s is null", name);
  if (!aligned(p, 16)) return fail(FG_ERR_ALIGN, "%s needs 16-byte alignment", name);
  return FG_OK;
}

}  // namespace

fg_status gemm(const GemmArgs& a, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (gemm_q4ts_supported(a)) return gemm_q4ts(a, ws, ws_bytes, st);
  if (a.dtype == FG_F16 && a.M >= 64 && a.quant) {
    // converted back to fp16 once into the workspace, then the dense product
    GemmArgs d = a;
    char* w = static_cast<char*>(ws);
    size_t used = 0;
    for (int i = 0; i < a.nseg; ++i) {
      const size_t bytes = up(static_cast<size_t>(a.K) * a.seg[i].N * 2);
      if (!ws || used + bytes > ws_bytes) return fail(FG_ERR_WORKSPACE, "workspace too small for the fp16 weight");
      FG_TRY(dequant_rows(a.seg[i].codes, a.seg[i].mins, a.seg[i].scales, a.K, a.seg[i].N, w + used, FG_F16, st));
      d.seg[i].dense = w + used;
      d.seg[i].codes = nullptr;
      d.seg[i].packed = nullptr;
      used += bytes;
    }
    d.quant = 0;
    if (gemm_tc_supported(d)) return gemm_tc(d, w + used, ws_bytes - used, st);
    return gemm_simt(d, st);
  }
  if (gemm_tc_supported(a)) return gemm_tc(a, ws, ws_bytes, st);
  return gemm_simt(a, st);
}

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, fg_dtype dt, int quant, bool packed) {
  if (dt != FG_F16 || M <= 0) return 0;
  if (quant && packed && M <= 256) return gemm_q4ts_workspace_bytes(M, N, K);
  if (M < 64) return 0;
  const size_t tc = gemm_tc_workspace_bytes(M, N, K);
  return quant ? up(static_cast<size_t>(K) * N * 2) + 3 * kAlign + tc : tc;
}

}  // namespace fg

using namespace fg;

extern "C" {

size_t fg_prefill_workspace_bytes(const fg_layer* L, int64_t b, int64_t s) {
  if (check_layer(L) != FG_OK || b < 0 || s < 0) return 0;
  return activations_bytes(*L, b * s) + scratch_bytes(*L, b * s, s, false);
}

size_t fg_decode_workspace_bytes(const fg_layer* L, int64_t b, int64_t capacity) {
  if (check_layer(L) != FG_OK || check_decode_copies(*L) != FG_OK || b < 0 || capacity < 0) return 0;
  return activations_bytes(*L, b) + scratch_bytes(*L, b, capacity, true);
}

size_t fg_prefill_block_workspace_bytes(const fg_layer* L, int64_t b, int64_t s) {
  if (check_layer(L) != FG_OK || b < 0 || s < 0) return 0;
  return fg_prefill_workspace_bytes(L, b, s) + 2 * up(b * s * L->h1 * dtype_bytes(L->dtype));
}

size_t fg_decode_block_workspace_bytes(const fg_layer* L, int64_t b, int64_t capacity) {
  if (check_layer(L) != FG_OK || b < 0 || capacity < 0) return 0;
  return fg_decode_workspace_bytes(L, b, capacity) + 2 * up(b * L->h1 * dtype_bytes(L->dtype));
}

size_t fg_linear_workspace_bytes(int64_t M, int64_t K, int64_t N, fg_codec codec, fg_dtype dtype) {
  if (M < 0 || K <= 0 || N <= 0) return 0;
  const int q = codec == FG_CODEC_Q4G64;
  const size_t a = gemm_workspace_bytes(M, N, K, dtype, q, true), b = gemm_workspace_bytes(M, N, K, dtype, q, false);
  return a > b ? a : b;
}

fg_status fg_linear(const fg_wmat* w, fg_codec codec, fg_dtype dtype, const void* x, int64_t M,
                    const void* r, int32_t relu, void* y, void* ws, size_t ws_bytes,
                    cudaStream_t stream) {
  if (!w) return fail(FG_ERR_ARG, "null weight");
  if (dtype != FG_F16 && dtype != FG_F32) return fail(FG_ERR_ARG, "dtype");
  if (codec != FG_CODEC_NONE && codec != FG_CODEC_Q4G64) return fail(FG_ERR_ARG, "codec");
  if (M < 0 || w->K <= 0 || w->N <= 0) return fail(FG_ERR_ARG, "sizes");
  if (w->K % 64 || w->N % 64) return fail(FG_ERR_SHAPE, "K and N must be multiples of 64");
  FG_TRY(check_wmat(*w, w->K, w->N, codec, "w"));
  if (M == 0) return FG_OK;
  FG_TRY(check_act(x, "x"));
  FG_TRY(check_act(y, "y"));
  if (r && !aligned(r, 16)) return fail(FG_ERR_ALIGN, "r needs 16-byte alignment");
  if (r == y || x == y) return fail(FG_ERR_ARG, "y must not alias x or r");
  const size_t need = fg_linear_workspace_bytes(M, w->K, w->N, codec, dtype);
  if (need && (!ws || ws_bytes < need)) return fail(FG_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  if (!aligned(ws, kAlign)) return fail(FG_ERR_ALIGN, "workspace needs 256-byte alignment");
  fg_layer L{};
  L.codec = codec;
  L.dtype = dtype;
  GemmArgs a = product(L, x, w->K, M, w, 1, y, w->N, r, w->N, relu ? 1 : 0);
  return gemm(a, ws, ws_bytes, stream);
}

size_t fg_pack_weight_bytes(int64_t K, int64_t N, int32_t format) {
  if (K <= 0 || N <= 0 || K % 64 || N % 128) return 0;
  if (format != FG_PACK_EXACT && format != FG_PACK_F16META) return 0;
  return pack_weight_bytes(K, N, format);
}

fg_status fg_pack_weight(const fg_wmat* w, int32_t format, uint8_t* packed, cudaStream_t stream) {
  if (!w || !w->codes || !w->mins || !w->scales || !packed) return fail(FG_ERR_ARG, "null weight arrays or packed buffer");
  if (format != FG_PACK_EXACT && format != FG_PACK_F16META) return fail(FG_ERR_ARG, "unknown pack format %d", format);
  if (w->K <= 0 || w->N <= 0) return fail(FG_ERR_ARG, "sizes");
  if (w->K % 64 || w->N % 128) return fail(FG_ERR_SHAPE, "K must be a multiple of 64 and N of 128");
  if (!aligned(w->codes, 16) || !aligned(packed, 16) || !aligned(w->mins, 4) || !aligned(w->scales, 4))
    return fail(FG_ERR_ALIGN, "codes and the packed buffer need 16-byte alignment");
  return pack_weight(w->codes, w->mins, w->scales, w->K, w->N, format, packed, stream);
}

size_t fg_decode_attention_workspace_bytes(const fg_kv* kv) {
  if (!kv || kv->b < 0 || kv->heads <= 0 || kv->head_dim <= 0 || kv->capacity <= 0) return 0;
  if (kv->codec != FG_CODEC_Q4G64 || kv->dtype != FG_F16) return 0;
  return decode_attention_workspace_bytes(kv->b, kv->heads, kv->head_dim, kv->capacity);
}

}  // extern "C"

namespace fg {
fg_status check_decode_attention(const fg_kv* kv, const void* q, int64_t ldq, int64_t pos, const void* out,
                                 int64_t ldo) {
  if (!kv) return fail(FG_ERR_ARG, "null kv");
  if (kv->heads <= 0 || kv->head_dim <= 0 || kv->b < 0) return fail(FG_ERR_ARG, "kv sizes");
  if (kv->head_dim != 64 && kv->head_dim != 128)
    return fail(FG_ERR_UNSUPPORTED, "head_dim %d (64 or 128)", kv->head_dim);
  FG_TRY(check_kv(kv, kv->b, kv->heads, kv->head_dim, kv->codec, kv->dtype));
  if (pos < 0 || pos >= kv->capacity)
    return fail(FG_ERR_CAPACITY, "pos %lld outside [0, %lld)", (long long)pos, (long long)kv->capacity);
  const int64_t h1 = static_cast<int64_t>(kv->heads) * kv->head_dim;
  if (ldq < h1 || ldo < h1 || ldq % 8 || ldo % 8) return fail(FG_ERR_SHAPE, "ldq/ldo must be >= h1 and multiples of 8");
  if (kv->b == 0) return FG_OK;
  FG_TRY(check_act(q, "q"));
  return check_act(out, "out");
}
}  // namespace fg

extern "C" {

fg_status fg_decode_attention(const fg_kv* kv, const void* q, int64_t ldq, int64_t pos, void* out,
                              int64_t ldo, void* ws, size_t ws_bytes, cudaStream_t stream) {
  FG_TRY(check_decode_attention(kv, q, ldq, pos, out, ldo));
  if (kv->b == 0) return FG_OK;
  const size_t need = fg_decode_attention_workspace_bytes(kv);
  if (need && (!ws || ws_bytes < need)) return fail(FG_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  if (need && !aligned(ws, 16)) return fail(FG_ERR_ALIGN, "workspace needs 16-byte alignment");
  return decode_attention(*kv, q, ldq, nullptr, nullptr, 0, kv->b, pos, out, ldo, ws, ws_bytes, stream);
}

fg_status fg_kv_append(const fg_kv* kv, const void* k_new, const void* v_new, int64_t pos,
                       cudaStream_t stream) {
  if (!kv) return fail(FG_ERR_ARG, "null kv");
  if (kv->heads <= 0 || kv->head_dim <= 0 || kv->b < 0) return fail(FG_ERR_ARG, "kv sizes");
  if (kv->head_dim % 64) return fail(FG_ERR_SHAPE, "head_dim must be a multiple of 64");
  FG_TRY(check_kv(kv, kv->b, kv->heads, kv->head_dim, kv->codec, kv->dtype));
  if (pos < 0 || pos >= kv->capacity)
    return fail(FG_ERR_CAPACITY, "pos %lld outside [0, %lld)", (long long)pos, (long long)kv->capacity);
  if (kv->b == 0) return FG_OK;
  FG_TRY(check_act(k_new, "k_new"));
  FG_TRY(check_act(v_new, "v_new"));
  const int64_t h1 = static_cast<int64_t>(kv->heads) * kv->head_dim;
  return kv_store(*kv, k_new, v_new, h1, kv->b, 1, pos, stream);
}

fg_status fg_prefill_layer(const fg_layer* L, const void* x, int64_t b, int64_t s, const fg_kv* kv,
                           void* y, void* ws, size_t ws_bytes, cudaStream_t stream) {
  FG_TRY(check_layer(L));
  if (b < 0 || s < 0) return fail(FG_ERR_ARG, "negative size");
  FG_TRY(check_kv(kv, b, L->heads, L->h1 / L->heads, L->codec, L->dtype));
  if (s > kv->capacity) return fail(FG_ERR_CAPACITY, "s %lld exceeds capacity %lld", (long long)s, (long long)kv->capacity);
  if (b == 0 || s == 0) return FG_OK;
  FG_TRY(check_act(x, "x"));
  FG_TRY(check_act(y, "y"));
  const size_t need = fg_prefill_workspace_bytes(L, b, s);
  if (!ws || ws_bytes < need)
    return fail(FG_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  if (!aligned(ws, kAlign)) return fail(FG_ERR_ALIGN, "workspace needs 256-byte alignment");
  return run_prefill(*L, x, b, s, *kv, y, ws, scratch_bytes(*L, b * s, s, false), stream);
}

fg_status fg_decode_step(const fg_layer* L, const void* t, int64_t b, int64_t pos, const fg_kv* kv,
                         void* y, void* ws, size_t ws_bytes, cudaStream_t stream) {
  FG_TRY(check_layer(L));
  FG_TRY(check_decode_copies(*L));
  if (b < 0) return fail(FG_ERR_ARG, "negative size");
  FG_TRY(check_kv(kv, b, L->heads, L->h1 / L->heads, L->codec, L->dtype));
  if (pos < 0 || pos >= kv->capacity)
    return fail(FG_ERR_CAPACITY, "pos %lld outside [0, %lld)", (long long)pos, (long long)kv->capacity);
  if (b == 0) return FG_OK;
  FG_TRY(check_act(t, "t"));
  FG_TRY(check_act(y, "y"));
  const size_t need = fg_decode_workspace_bytes(L, b, kv->capacity);
  if (!ws || ws_bytes < need)
    return fail(FG_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  if (!aligned(ws, kAlign)) return fail(FG_ERR_ALIGN, "workspace needs 256-byte alignment");
  return run_decode(*L, t, b, pos, *kv, y, ws, scratch_bytes(*L, b, kv->capacity, true), stream);
}

fg_status fg_prefill_block(const fg_layer* layers, int32_t l, const void* x, int64_t b, int64_t s,
                           const fg_kv* kvs, void* y, void* ws, size_t ws_bytes,
                           cudaStream_t stream) {
  if (!layers || !kvs || l <= 0) return fail(FG_ERR_ARG, "layers/kvs/l");
  for (int32_t i = 0; i < l; ++i) {
    FG_TRY(check_layer(&layers[i]));
    if (layers[i].h1 != layers[0].h1 || layers[i].dtype != layers[0].dtype)
      return fail(FG_ERR_SHAPE, "layers differ in h1/dtype");
    FG_TRY(check_kv(&kvs[i], b, layers[i].heads, layers[i].h1 / layers[i].heads, layers[i].codec,
                    layers[i].dtype));
    if (s > kvs[i].capacity) return fail(FG_ERR_CAPACITY, "s exceeds capacity");
  }
  if (b == 0 || s == 0) return FG_OK;
  FG_TRY(check_act(x, "x"));
  FG_TRY(check_act(y, "y"));
  size_t layer_ws = 0;
  for (int32_t i = 0; i < l; ++i) {
    const size_t w = fg_prefill_workspace_bytes(&layers[i], b, s);
    layer_ws = w > layer_ws ? w : layer_ws;
  }
  const size_t act = up(b * s * layers[0].h1 * dtype_bytes(layers[0].dtype));
  const size_t need = up(layer_ws) + 2 * act;
  if (!ws || ws_bytes < need) return fail(FG_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  if (!aligned(ws, kAlign)) return fail(FG_ERR_ALIGN, "workspace needs 256-byte alignment");
  char* ping[2] = {static_cast<char*>(ws) + up(layer_ws), static_cast<char*>(ws) + up(layer_ws) + act};
  const void* in = x;
  for (int32_t i = 0; i < l; ++i) {
    void* out = (i == l - 1) ? y : ping[i & 1];
    FG_TRY(run_prefill(layers[i], in, b, s, kvs[i], out, ws,
                       scratch_bytes(layers[i], b * s, s, false), stream));
    in = out;
  }
  return FG_OK;
}

fg_status fg_decode_block_step(const fg_layer* layers, int32_t l, const void* t, int64_t b,
                               int64_t pos, const fg_kv* kvs, void* y, void* ws, size_t ws_bytes,
                               cudaStream_t stream) {
  if (!layers || !kvs || l <= 0) return fail(FG_ERR_ARG, "layers/kvs/l");
  for (int32_t i = 0; i < l; ++i) {
    FG_TRY(check_layer(&layers[i]));
    FG_TRY(check_decode_copies(layers[i]));
    if (layers[i].h1 != layers[0].h1 || layers[i].h2 != layers[0].h2 || layers[i].dtype != layers[0].dtype)
      return fail(FG_ERR_SHAPE, "layers differ in h1/h2/dtype");
    FG_TRY(check_kv(&kvs[i], b, layers[i].heads, layers[i].h1 / layers[i].heads, layers[i].codec,
                    layers[i].dtype));
    if (pos < 0 || pos >= kvs[i].capacity)
      return fail(FG_ERR_CAPACITY, "pos %lld outside [0, %lld)", (long long)pos, (long long)kvs[i].capacity);
  }
  if (b == 0) return FG_OK;
  FG_TRY(check_act(t, "t"));
  FG_TRY(check_act(y, "y"));
  size_t layer_ws = 0;
  for (int32_t i = 0; i < l; ++i) {
    const size_t w = fg_decode_workspace_bytes(&layers[i], b, kvs[i].capacity);
    layer_ws = w > layer_ws ? w : layer_ws;
  }
  const size_t act = up(b * layers[0].h1 * dtype_bytes(layers[0].dtype));
  const size_t need = up(layer_ws) + 2 * act;
  if (!ws || ws_bytes < need) return fail(FG_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  if (!aligned(ws, kAlign)) return fail(FG_ERR_ALIGN, "workspace needs 256-byte alignment");
  char* ping[2] = {static_cast<char*>(ws) + up(layer_ws), static_cast<char*>(ws) + up(layer_ws) + act};
  const void* in = t;
  for (int32_t i = 0; i < l; ++i) {
    void* out = (i == l - 1) ? y : ping[i & 1];
    FG_TRY(run_decode(layers[i], in, b, pos, kvs[i], out, ws,
                      scratch_bytes(layers[i], b, kvs[i].capacity, true), stream));
    in = out;
  }
  return FG_OK;
}

// ---------------------------------------------------------------------------
// Decode with the weights offloaded to host memory (FlexGen notes, "4. 卸载
// 策略", Algorithm 1: the next layer's weights are loaded while the current
// layer computes).  On GB300 host memory is the Grace LPDDR behind
// NVLink-C2C.  The six decode copies of a layer are the only weight bytes a
// decode step reads; they go, layer by layer, into one of two device stage
// buffers on a copy stream, while the compute stream runs the previous
// layer from the other buffer.  Two events per buffer order the pair: the
// compute stream waits until a buffer is loaded, the copy stream until the
// layer that last read it has finished.
// ---------------------------------------------------------------------------
namespace {

struct StageLayout {
  size_t off[6];
  size_t bytes[6];
  size_t total;
};

StageLayout stage_layout(const fg_layer& L) {
  StageLayout S;
  const fg_wmat* m[6] = {&L.wq, &L.wk, &L.wv, &L.wo, &L.w1, &L.w2};
  size_t at = 0;
  for (int i = 0; i < 6; ++i) {
    S.off[i] = at;
    S.bytes[i] = pack_weight_bytes(m[i]->K, m[i]->N, m[i]->packed_format);
    at += up(S.bytes[i]);
  }
  S.total = at;
  return S;
}

struct OffloadEvents {
  cudaEvent_t loaded[2] = {nullptr, nullptr};
  cudaEvent_t released[2] = {nullptr, nullptr};
};

fg_status offload_events(OffloadEvents** out) {
  static std::mutex mu;
  static OffloadEvents ev[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(FG_ERR_CUDA, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(mu);
  OffloadEvents& e = ev[dev];
  for (int i = 0; i < 2; ++i) {
    if (!e.loaded[i] && cudaEventCreateWithFlags(&e.loaded[i], cudaEventDisableTiming) != cudaSuccess)
      return check_launch("cudaEventCreateWithFlags");
    if (!e.released[i] && cudaEventCreateWithFlags(&e.released[i], cudaEventDisableTiming) != cudaSuccess)
      return check_launch("cudaEventCreateWithFlags");
  }
  *out = &e;
  return FG_OK;
}

}  // namespace

extern "C" size_t fg_offload_stage_bytes(const fg_layer* L) {
  if (check_layer(L) != FG_OK || !decode_needs_copies(*L)) return 0;
  return 2 * stage_layout(*L).total;
}

extern "C" fg_status fg_decode_block_step_offload(const fg_layer* layers, int32_t l, const void* t, int64_t b,
                                                  int64_t pos, const fg_kv* kvs, void* y, void* ws, size_t ws_bytes,
                                                  void* stage, size_t stage_bytes, cudaStream_t stream,
                                                  cudaStream_t copy_stream) {
  if (!layers || !kvs || l <= 0) return fail(FG_ERR_ARG, "layers/kvs/l");
  for (int32_t i = 0; i < l; ++i) {
    FG_TRY(check_layer(&layers[i]));
    if (!decode_needs_copies(layers[i]))
      return fail(FG_ERR_UNSUPPORTED, "offloaded decode streams the decode copies of fp16 4-bit layers");
    FG_TRY(check_decode_copies(layers[i]));
    if (layers[i].h1 != layers[0].h1 || layers[i].h2 != layers[0].h2 ||
        layers[i].wq.packed_format != layers[0].wq.packed_format)
      return fail(FG_ERR_SHAPE, "layers differ in h1/h2/decode-copy format");
    FG_TRY(check_kv(&kvs[i], b, layers[i].heads, layers[i].h1 / layers[i].heads, layers[i].codec,
                    layers[i].dtype));
    if (pos < 0 || pos >= kvs[i].capacity)
      return fail(FG_ERR_CAPACITY, "pos %lld outside [0, %lld)", (long long)pos, (long long)kvs[i].capacity);
  }
  const StageLayout S = stage_layout(layers[0]);
  if (!stage || stage_bytes < 2 * S.total) return fail(FG_ERR_WORKSPACE, "stage %zu < %zu bytes", stage_bytes, 2 * S.total);
  if (!aligned(stage, kAlign)) return fail(FG_ERR_ALIGN, "stage needs 256-byte alignment");
  if (b == 0) return FG_OK;
  FG_TRY(check_act(t, "t"));
  FG_TRY(check_act(y, "y"));
  size_t layer_ws = 0;
  for (int32_t i = 0; i < l; ++i) {
    const size_t w = fg_decode_workspace_bytes(&layers[i], b, kvs[i].capacity);
    layer_ws = w > layer_ws ? w : layer_ws;
  }
  const size_t act = up(b * layers[0].h1 * dtype_bytes(layers[0].dtype));
  const size_t need = up(layer_ws) + 2 * act;
  if (!ws || ws_bytes < need) return fail(FG_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  if (!aligned(ws, kAlign)) return fail(FG_ERR_ALIGN, "workspace needs 256-byte alignment");

  OffloadEvents* E = nullptr;
  FG_TRY(offload_events(&E));
  char* buf[2] = {static_cast<char*>(stage), static_cast<char*>(stage) + S.total};
  // layer j's six decode copies into buffer j % 2, once the layer that last
  // read that buffer has finished
  auto load = [&](int32_t j) -> fg_status {
    const int s = j & 1;
    if (cudaStreamWaitEvent(copy_stream, E->released[s], 0) != cudaSuccess) return check_launch("cudaStreamWaitEvent");
    const fg_wmat* m[6] = {&layers[j].wq, &layers[j].wk, &layers[j].wv, &layers[j].wo, &layers[j].w1, &layers[j].w2};
    for (int k = 0; k < 6; ++k)
      if (cudaMemcpyAsync(buf[s] + S.off[k], m[k]->packed, S.bytes[k], cudaMemcpyDefault, copy_stream) != cudaSuccess)
        return check_launch("cudaMemcpyAsync (decode copy to the stage)");
    if (cudaEventRecord(E->loaded[s], copy_stream) != cudaSuccess) return check_launch("cudaEventRecord");
    return FG_OK;
  };
  char* ping[2] = {static_cast<char*>(ws) + up(layer_ws), static_cast<char*>(ws) + up(layer_ws) + act};
  const void* in = t;
  FG_TRY(load(0));
  for (int32_t i = 0; i < l; ++i) {
    if (i + 1 < l) FG_TRY(load(i + 1));   // the next layer streams in while this one computes
    const int s = i & 1;
    if (cudaStreamWaitEvent(stream, E->loaded[s], 0) != cudaSuccess) return check_launch("cudaStreamWaitEvent");
    fg_layer Ld = layers[i];   // the same layer, its decode copies read from the stage
    fg_wmat* m[6] = {&Ld.wq, &Ld.wk, &Ld.wv, &Ld.wo, &Ld.w1, &Ld.w2};
    for (int k = 0; k < 6; ++k) m[k]->packed = reinterpret_cast<const uint8_t*>(buf[s] + S.off[k]);
    void* out = (i == l - 1) ? y : ping[i & 1];
    FG_TRY(run_decode(Ld, in, b, pos, kvs[i], out, ws, scratch_bytes(Ld, b, kvs[i].capacity, true), stream));
    if (cudaEventRecord(E->released[s], stream) != cudaSuccess) return check_launch("cudaEventRecord");
    in = out;
  }
  return FG_OK;
}

}  // extern "C"
