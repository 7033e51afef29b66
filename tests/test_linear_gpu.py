"""GPU parity of fg_linear, the layer's dequant-fused product y = act(x.w + r)
(FlexGen notes, "背景知识" products, "5. 近似方法" weights stored in 4-bit
groups and converted back to FP16 before compute), against the oracle: x in
fp64 times the oracle's dequantized weights.

The fp16 tensor-core path accumulates in fp32 and rounds the output to fp16,
so each output is within a few fp16 ulps: bar max|d|/max|ref| <= 2e-3 for
every path, dense or 4-bit, with the default decode copy of a weight (the
stored fp32 (min, scale)) or with the opt-in fp16-metadata copy (compared
with that format's own oracle reading)."""
import numpy as np
import pytest
import torch

import synth
from oracle import codec as ocodec
from oracle import layer as olayer

EXACT, F16META = 0, 1


def _weight_ref(w16, fmt):
    """The weights a product multiplies by, per the oracle: the format of
    record's fp16(fmaf(q, scale, min)), or the fp16-metadata reading."""
    a = w16.cpu().numpy()
    if fmt == F16META:
        c, m, s = ocodec.quantize_g64(a)
        return ocodec.dequant_g64_f16meta(c, m, s).astype(np.float64)
    return olayer.weight_for_compute(a, True, "f16" if w16.dtype == torch.float16 else "f32")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fg():
    import int4_group_quantized_gb300 as fg
    return fg


CASES = [
    # (M, K, N, quantized, relu, residual, dtype)
    (64, 4096, 12288, True, False, False, torch.float16),     # decode QKV, 6.7B
    (64, 4096, 4096, True, False, True, torch.float16),       # decode O + residual (split over K)
    (64, 4096, 16384, True, True, False, torch.float16),      # decode FC1 + relu
    (64, 16384, 4096, True, False, True, torch.float16),      # decode FC2 (long K)
    (100, 512, 768, True, True, True, torch.float16),         # ragged block, 128-wide tiles
    (256, 1024, 512, True, False, True, torch.float16),       # b = 256: two 128-row tiles per CTA
    (200, 768, 2304, True, False, False, torch.float16),
    (385, 256, 512, False, False, True, torch.float16),       # prefill-like, dense fp16 weights
    (1000, 512, 768, False, True, False, torch.float16),
    (4096, 1024, 1024, False, False, True, torch.float16),
    (5, 128, 64, True, True, True, torch.float16),            # small block: CUDA cores
    (32, 768, 2304, True, False, False, torch.float16),
    (7, 256, 192, True, False, True, torch.float32),          # fp32 activations
    (1, 4096, 4096, True, False, True, torch.float16),        # one sequence (GEMV shape)
    (33, 2048, 1536, True, True, False, torch.float16),       # ragged 64-row block
    (64, 64, 1024, True, False, False, torch.float16),        # a single k tile
    (130, 4096, 256, True, False, True, torch.float16),       # two tiles, eight K splits
    # odd k-tile counts: splits whose last two-tile chunk holds one tile
    (64, 960, 512, True, False, True, torch.float16),         # 15 k tiles, 64-row block
    (96, 1088, 768, True, True, False, torch.float16),        # 17 k tiles, 128-row block
    (256, 960, 384, True, False, True, torch.float16),        # 15 k tiles, 256-row block
    # blocks of a few sequences (padded to the kernel's 32-row MMA)
    (2, 768, 2304, True, False, False, torch.float16),        # OPT-125M QKV, two sequences
    (3, 4096, 4096, True, False, True, torch.float16),
    (4, 16384, 4096, True, False, True, torch.float16),       # long K: sixteen splits
    (6, 1024, 768, True, True, False, torch.float16),
    (8, 4096, 16384, True, True, False, torch.float16),
    (8, 1088, 512, True, False, True, torch.float16),         # 17 k tiles: ragged warp ranges
    (1, 12288, 256, True, False, False, torch.float16),       # a single channel tile, no split of N
]

# quantized fp16 products with at most 256 rows run on the decode-copy
# kernel when the weight carries its copy (in either format), on the
# converted-weight tensor-core path (M >= 64) or the CUDA cores otherwise;
# all are checked
PACKED = [c + (fmt,) for c in CASES if c[3] and c[6] == torch.float16 and c[0] <= 256 and c[2] % 128 == 0
          for fmt in (EXACT, F16META)]
ALL = [c + (None,) for c in CASES] + PACKED


@pytest.mark.parametrize("case", ALL, ids=lambda c: "M%d_K%d_N%d_%s%s%s_%s%s" % (
    c[0], c[1], c[2], "q4" if c[3] else "dense", "_relu" if c[4] else "", "_res" if c[5] else "",
    "f16" if c[6] == torch.float16 else "f32", {None: "", EXACT: "_packed", F16META: "_packed16"}[c[7]]))
def test_linear_matches_oracle(fg, case):
    M, K, N, quant, relu, res, dt, fmt = case
    w16 = synth.normal((K, N), 7 + K + N, synth.WEIGHT_STD, dt, "cuda")
    x = synth.normal((M, K), 11 + M, 1.0, dt, "cuda")
    r = synth.normal((M, N), 13 + M, 1.0, dt, "cuda") if res else None
    if quant:
        W = fg.QuantWeight.from_dense(w16, True, pack=fmt is not None, pack_format=fmt or 0)
        wref = _weight_ref(w16, fmt or EXACT)
    else:
        W = fg.QuantWeight.from_dense(w16, False)
        wref = w16.cpu().numpy().astype(np.float64)
    y = torch.empty((M, N), dtype=dt, device="cuda")
    fg.fg_linear(W, x, y, r, relu)
    fg.fg_sync_status()
    ref = x.cpu().numpy().astype(np.float64) @ wref
    if res:
        ref = ref + r.cpu().numpy().astype(np.float64)
    if relu:
        ref = np.maximum(ref, 0)
    got = y.cpu().numpy().astype(np.float64)
    tol = 2e-3 if dt == torch.float16 else 1e-5
    err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert err <= tol, f"rel err {err}"


@pytest.mark.parametrize("fmt", [None, EXACT, F16META])
def test_linear_repeatable(fg, fmt):
    """Two calls give identical bits (no atomics in the reduction order)."""
    w16 = synth.normal((4096, 4096), 3, synth.WEIGHT_STD, torch.float16, "cuda")
    W = fg.QuantWeight.from_dense(w16, True, pack=fmt is not None, pack_format=fmt or 0)
    x = synth.normal((64, 4096), 4, 1.0, torch.float16, "cuda")
    y1 = torch.empty((64, 4096), dtype=torch.float16, device="cuda")
    y2 = torch.empty_like(y1)
    fg.fg_linear(W, x, y1)
    fg.fg_linear(W, x, y2)
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("M", [1, 3, 8, 32, 64, 128, 256])
@pytest.mark.parametrize("fmt", [EXACT, F16META])
def test_decode_product_restores_weights_bit_exactly(fg, M, fmt):
    """With one-hot rows x = e_k the product returns weight row k itself
    (one nonzero term per output, exact in fp32, already an fp16 value): the
    decode copy's conversion gives exactly the oracle's weights -- the
    format of record's fp16(fmaf(q, scale, min)), or the fp16-metadata
    reading -- at every k tile and K split."""
    K, N = 4096, 12288 if M <= 64 else 1024
    w16 = synth.normal((K, N), 17, synth.WEIGHT_STD, torch.float16, "cuda")
    W = fg.QuantWeight.from_dense(w16, True, pack=True, pack_format=fmt)
    ks = (np.arange(M) * 4099 + 5) % K          # spread over k tiles and splits
    x = torch.zeros((M, K), dtype=torch.float16)
    x[np.arange(M), ks] = 1.0
    x = x.cuda()
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    fg.fg_linear(W, x, y)
    fg.fg_sync_status()
    c, m, s = (t.cpu().numpy() for t in (W.codes, W.mins, W.scales))
    rows = (ocodec.dequant_g64_f16meta(c[ks], m[ks], s[ks]) if fmt == F16META
            else ocodec.dequant_g64(c[ks], m[ks], s[ks], np.float16))
    got = y.cpu().numpy()
    assert np.array_equal(got.view(np.uint16), rows.view(np.uint16)), \
        f"{np.mean(got != rows)} of the weights differ"


@pytest.mark.parametrize("fmt", [EXACT, F16META])
def test_pack_layout(fg, fmt):
    """fg_pack_weight's layout as its declaration states it, rebuilt here in
    numpy from the [K][N/2] codes and [K][N/64] (min, scale): one block per
    (128-channel tile, 64-k tile), 5120 bytes (fp32 pairs) or 4608 (fp16
    pairs).  Codes in 16-byte units [q][g2][t]: word w is channel
    32q + t/4 + 8w, k pairs j = 16 g2 + 4e + t%4 with k = 2j in nibble slot e
    and k = 2j+1 in slot e+4.  fp32 pairs: unit gl*512 + j*16 holds (scale,
    scale', min, min') of k pair j; fp16 pairs: units [gl][u][c4] hold
    (scale, scale') and (min, min') for the k pairs j = 8u + c4 and
    8u + 4 + c4."""
    K, N = 192, 384
    B = 5120 if fmt == EXACT else 4608
    w16 = synth.normal((K, N), 5, synth.WEIGHT_STD, torch.float16, "cuda")
    W = fg.QuantWeight.from_dense(w16, True, pack=True, pack_format=fmt)
    fg.fg_sync_status()
    codes = W.codes.cpu().numpy()
    nib = np.empty((K, N), dtype=np.uint32)
    nib[:, 0::2] = codes & 15
    nib[:, 1::2] = codes >> 4
    sc32, mn32 = W.scales.cpu().numpy(), W.mins.cpu().numpy()
    sc = sc32.astype(np.float16)    # [K][N/64], rounded to nearest even
    mn = mn32.astype(np.float16)
    packed = W.packed.cpu().numpy()
    assert packed.size == (K // 64) * (N // 128) * B == fg.fg_pack_weight_bytes(K, N, fmt)
    blocks = packed.reshape(N // 128, K // 64, B)
    lane = np.arange(32)
    for t in range(N // 128):
        for u in range(K // 64):
            blk = blocks[t, u]
            cw = blk[:4096].view(np.uint32).reshape(4, 2, 32, 4)
            for q in range(4):
                for g2 in range(2):
                    for w in range(4):
                        n = 128 * t + 32 * q + lane // 4 + 8 * w           # per lane
                        want = np.zeros(32, dtype=np.uint32)
                        for e in range(4):
                            k = 64 * u + 2 * (16 * g2 + 4 * e + lane % 4)
                            want |= nib[k, n] << np.uint32(4 * e)
                            want |= nib[k + 1, n] << np.uint32(4 * (e + 4))
                        assert np.array_equal(cw[q, g2, :, w], want), (t, u, q, g2, w)
            if fmt == EXACT:
                pr = blk[4096:].view(np.float32).reshape(2, 32, 4)     # [gl][j][s, s', m, m']
                for gl in range(2):
                    g = 2 * t + gl
                    for j in range(32):
                        k = 64 * u + 2 * j
                        want = np.array([sc32[k, g], sc32[k + 1, g], mn32[k, g], mn32[k + 1, g]], np.float32)
                        assert np.array_equal(pr[gl, j].view(np.uint32), want.view(np.uint32)), (t, u, gl, j)
                continue
            pr = blk[4096:].view(np.uint16).reshape(2, 4, 4, 2, 4)   # [gl][u][c4][hi][s, s', m, m']
            for gl in range(2):
                g = 2 * t + gl
                for uu in range(4):
                    for c4 in range(4):
                        for hi in range(2):
                            k = 64 * u + 2 * (8 * uu + 4 * hi + c4)
                            got = pr[gl, uu, c4, hi]
                            want = np.array([sc[k, g], sc[k + 1, g], mn[k, g], mn[k + 1, g]]).view(np.uint16)
                            assert np.array_equal(got, want), (t, u, gl, uu, c4, hi)
