"""Failure handling on the GPU without faulting it: every bounded wait of the
tensor-core kernels gives up after a host-set number of polls
(fg_set_wait_limit), sets the library's device error word and lets its CTA
leave once its own copies and MMAs in flight have completed and its tensor
memory is freed.  A limit of 0 makes every such wait give up at once (a
dependency that never arrives); the host then reads FG_ERR_DEVICE_TIMEOUT
from fg_sync_status, and the next call with the default limit is correct.

The products are checked against the oracle (x in fp64 times the oracle's
dequantized weights) at the product tests' bar, 2e-3 of the largest output."""
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


@pytest.mark.parametrize("M,quant", [(64, True), (128, False)], ids=["decode_copy_M64", "dense_M128"])
def test_wait_timeout_is_reported_and_the_library_recovers(fg, M, quant):
    K, N = 4096, 4096
    w16 = synth.normal((K, N), 51, synth.WEIGHT_STD, torch.float16, "cuda")
    W = fg.QuantWeight.from_dense(w16, quant, pack=quant or None)
    x = synth.normal((M, K), 52, 1.0, torch.float16, "cuda")
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = fg.workspace(max(fg.fg_linear_workspace_bytes(M, K, N, quant, torch.float16), 1), "cuda")
    fg.fg_sync_status()
    prev = fg.fg_set_wait_limit(0)
    try:
        fg.fg_linear(W, x, y, ws=ws)
        with pytest.raises(fg.FGError) as e:
            fg.fg_sync_status()
        assert e.value.status == 7, e.value            # FG_ERR_DEVICE_TIMEOUT
    finally:
        assert fg.fg_set_wait_limit(prev) == 0
    fg.fg_sync_status()                                # the error word was cleared
    fg.fg_linear(W, x, y, ws=ws)
    fg.fg_sync_status()
    wref = (olayer.weight_for_compute(w16.cpu().numpy(), True, "f16") if quant
            else w16.cpu().numpy().astype(np.float64))
    ref = x.cpu().numpy().astype(np.float64) @ wref
    err = np.max(np.abs(y.cpu().numpy().astype(np.float64) - ref)) / np.max(np.abs(ref))
    assert err <= 2e-3, f"rel err {err} after recovery"


def test_topk_attention_wait_timeout_is_reported_and_recovers(fg):
    """The top-K attention kernel stages K with bulk copies behind bounded
    mbarrier waits: with a limit of 0 they give up, the CTA drains its copies
    and raises the error word; with the default limit the call is correct
    (against the oracle, as in test_topk_gpu.py)."""
    b, H, d, length, keep = 2, 2, 128, 600, 60   # three staged chunks
    h1 = H * d
    kv = fg.KVCache(b, H, d, length, True, torch.float16, "cuda")
    k = synth.normal((length, b, h1), 81, 1.3, torch.float16, "cuda")
    v = synth.normal((length, b, h1), 82, 1.3, torch.float16, "cuda")
    for p in range(length):
        fg.fg_kv_append(kv, k[p].contiguous(), v[p].contiguous(), p)
    q = synth.normal((b, h1), 83, 1.3, torch.float16, "cuda")
    out = torch.empty_like(q)
    fg.fg_sync_status()
    prev = fg.fg_set_wait_limit(0)
    try:
        fg.fg_decode_attention_topk(kv, q, length - 1, keep, out)
        with pytest.raises(fg.FGError) as e:
            fg.fg_sync_status()
        assert e.value.status == 7, e.value
    finally:
        assert fg.fg_set_wait_limit(prev) == 0
    fg.fg_sync_status()
    fg.fg_decode_attention_topk(kv, q, length - 1, keep, out)
    fg.fg_sync_status()
    oc = olayer.KVCache(b, H, d, length, True, "f16")
    oc.store(k.cpu().numpy().astype(np.float64).transpose(1, 0, 2),
             v.cpu().numpy().astype(np.float64).transpose(1, 0, 2), 0)
    want, _ = olayer.attention_topk(q.cpu().numpy().astype(np.float64).reshape(b, H, d), oc.k_val, oc.v_val, keep)
    got = out.cpu().numpy().astype(np.float64).reshape(b, H, d)
    assert np.max(np.abs(got - want)) / np.max(np.abs(want)) <= 5e-3

