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
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "M%d_K%d_N%d_%s%s%s_%s" % (
    c[0], c[1], c[2], "q4" if c[3] else "dense", "_relu" if c[4] else "", "_res" if c[5] else "",
    "f16" if c[6] == torch.float16 else "f32"))
def test_linear_matches_oracle(fg, case):
    M, K, N, quant, relu, res, dt = case
    w16 = synth.normal((K, N), 7 + K + N, synth.WEIGHT_STD, dt, "cuda")
    x = synth.normal((M, K), 11 + M, 1.0, dt, "cuda")
    r = synth.normal((M, N), 13 + M, 1.0, dt, "cuda") if res else None
    if quant:
        W = fg.QuantWeight.from_dense(w16, True)
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


def test_linear_repeatable(fg):
    """Two calls give identical bits (no atomics in the reduction order)."""
    w16 = synth.normal((4096, 4096), 3, synth.WEIGHT_STD, torch.float16, "cuda")
    W = fg.QuantWeight.from_dense(w16, True)
    x = synth.normal((64, 4096), 4, 1.0, torch.float16, "cuda")
    y1 = torch.empty((64, 4096), dtype=torch.float16, device="cuda")
    y2 = torch.empty_like(y1)
    fg.fg_linear(W, x, y1)
    fg.fg_linear(W, x, y2)
    assert torch.equal(y1, y2)
