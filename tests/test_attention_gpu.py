"""GPU parity of fg_decode_attention (FlexGen notes, "背景知识": decode
attention Softmax(t_Q x_K^T / sqrt(h1)) x_V over the cache; "5. 近似方法": K/V
stored in 4-bit groups along the hidden dimension) against the oracle's
attention over the same cache contents.

The cache is filled through fg_kv_append (bit-exact against the oracle's
codec, see test_codec_gpu.py), so both sides attend over identical values;
the bar covers the fp16 query and fp32 accumulation: max|d|/max|ref| <= 5e-3
for fp16, 1e-5 for fp32."""
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
    # (b, heads, head_dim, filled slots, capacity, quantized, dtype)
    (2, 4, 128, 300, 320, True, torch.float16),    # few (sequence, head) pairs: split over tokens
    (3, 2, 64, 101, 101, True, torch.float16),     # ragged tail, pos = capacity - 1
    (16, 8, 128, 530, 544, True, torch.float16),   # many pairs: no split
    (1, 1, 64, 1, 8, True, torch.float16),         # a single cached token
    (2, 2, 64, 37, 40, True, torch.float32),       # fp32 activations: CUDA-core kernel
    (2, 2, 128, 37, 40, False, torch.float16),     # uncompressed cache
    (4, 2, 128, 333, 333, True, torch.float16),    # capacity not a multiple of 4: register-block kernel
    (2, 3, 128, 70, 72, True, torch.float16),      # ragged last chunk of the shared-memory ring
    (1, 2, 128, 1000, 1024, True, torch.float16),  # 16 token splits of 64, one ring chunk each
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b%d_H%d_d%d_len%d_%s_%s" % (
    c[0], c[1], c[2], c[3], "q4" if c[5] else "dense", "f16" if c[6] == torch.float16 else "f32"))
def test_decode_attention_matches_oracle(fg, case):
    b, H, d, length, cap, quant, dt = case
    h1 = H * d
    kv = fg.KVCache(b, H, d, cap, quant, dt, "cuda")
    ocache = olayer.KVCache(b, H, d, cap, quant, "f16" if dt == torch.float16 else "f32")
    k = synth.normal((length, b, h1), 21 + length, 1.3, dt, "cuda")
    v = synth.normal((length, b, h1), 22 + length, 1.3, dt, "cuda")
    for p in range(length):
        fg.fg_kv_append(kv, k[p].contiguous(), v[p].contiguous(), p)
    ocache.store(k.cpu().numpy().astype(np.float64).transpose(1, 0, 2),
                 v.cpu().numpy().astype(np.float64).transpose(1, 0, 2), 0)
    q = synth.normal((b, h1), 23, 1.3, dt, "cuda")
    out = torch.empty((b, h1), dtype=dt, device="cuda")
    fg.fg_decode_attention(kv, q, length - 1, out)
    fg.fg_sync_status()
    ref = olayer.attention(q.cpu().numpy().astype(np.float64).reshape(b, 1, H, d), ocache.k_val[:, :, :length],
                           ocache.v_val[:, :, :length], np.array([length - 1])).reshape(b, h1)
    tol = 5e-3 if dt == torch.float16 else 1e-5
    err = np.max(np.abs(out.cpu().numpy().astype(np.float64) - ref)) / np.max(np.abs(ref))
    assert err <= tol, f"rel err {err}"


def test_decode_attention_errors(fg):
    kv = fg.KVCache(2, 2, 64, 8, True, torch.float16, "cuda")
    q = torch.zeros((2, 128), dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(fg.FGError) as e:
        fg.fg_decode_attention(kv, q, 8, out)
    assert e.value.status == 4
