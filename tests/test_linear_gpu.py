"""GPU parity of fg_linear, the layer's dequant-fused product y = act(x.w + r)
(FlexGen notes, "背景知识" products, "5. 近似方法" weights stored in 4-bit
groups and converted back to FP16 before compute), against the oracle: x in
fp64 times the oracle's dequantized weights.

The fp16 tensor-core path accumulates in fp32 and rounds the output to fp16,
so each output is within a few fp16 ulps: bar max|d|/max|ref| <= 2e-3."""
import numpy as np
import pytest
import torch

import synth
from oracle import layer as olayer

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
]

# quantized fp16 products with at most 256 rows run on the packed-weight
# kernel when the weight carries its channel-major copy, on the shared-memory
# kernel otherwise; both are checked
PACKED = [c + (True,) for c in CASES if c[3] and c[6] == torch.float16 and c[0] <= 256 and c[2] % 128 == 0]
ALL = [c + (False,) for c in CASES] + PACKED


@pytest.mark.parametrize("case", ALL, ids=lambda c: "M%d_K%d_N%d_%s%s%s_%s%s" % (
    c[0], c[1], c[2], "q4" if c[3] else "dense", "_relu" if c[4] else "", "_res" if c[5] else "",
    "f16" if c[6] == torch.float16 else "f32", "_packed" if c[7] else ""))
def test_linear_matches_oracle(fg, case):
    M, K, N, quant, relu, res, dt, packed = case
    w16 = synth.normal((K, N), 7 + K + N, synth.WEIGHT_STD, dt, "cuda")
    x = synth.normal((M, K), 11 + M, 1.0, dt, "cuda")
    r = synth.normal((M, N), 13 + M, 1.0, dt, "cuda") if res else None
    if quant:
        W = fg.QuantWeight.from_dense(w16, True, pack=packed)
        wref = olayer.weight_for_compute(w16.cpu().numpy(), True, "f16" if dt == torch.float16 else "f32")
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


@pytest.mark.parametrize("packed", [False, True])
def test_linear_repeatable(fg, packed):
    """Two calls give identical bits (no atomics in the reduction order)."""
    w16 = synth.normal((4096, 4096), 3, synth.WEIGHT_STD, torch.float16, "cuda")
    W = fg.QuantWeight.from_dense(w16, True, pack=packed)
    x = synth.normal((64, 4096), 4, 1.0, torch.float16, "cuda")
    y1 = torch.empty((64, 4096), dtype=torch.float16, device="cuda")
    y2 = torch.empty_like(y1)
    fg.fg_linear(W, x, y1)
    fg.fg_linear(W, x, y2)
    assert torch.equal(y1, y2)


def test_pack_layout(fg):
    """fg_pack_weight's layout as its declaration states it, rebuilt here in
    numpy from the [K][N/2] codes and [K][N/64] (min, scale): 4608-byte
    blocks per (128-channel tile, 64-k tile).  Codes in 16-byte units
    [q][g2][t]: word w is channel 32q + t/4 + 8w, k pairs j = 16 g2 + 4e + t%4
    with k = 2j in nibble slot e and k = 2j+1 in slot e+4.  Then per group
    16-byte units [u][c4]: fp16 (scale, scale') and (min, min') for the k
    pairs j = 8u + c4 and 8u + 4 + c4."""
    K, N = 192, 384
    w16 = synth.normal((K, N), 5, synth.WEIGHT_STD, torch.float16, "cuda")
    W = fg.QuantWeight.from_dense(w16, True, pack=True)
    fg.fg_sync_status()
    codes = W.codes.cpu().numpy()
    nib = np.empty((K, N), dtype=np.uint32)
    nib[:, 0::2] = codes & 15
    nib[:, 1::2] = codes >> 4
    sc = W.scales.cpu().numpy().astype(np.float16)    # [K][N/64], rounded to nearest even
    mn = W.mins.cpu().numpy().astype(np.float16)
    packed = W.packed.cpu().numpy()
    assert packed.size == K * N // 2 + K * N // 16
    blocks = packed.reshape(N // 128, K // 64, 4608)
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
