"""fg_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory (code embedded in an application that owns the GPU
memory pool, or a loop that cannot afford the synchronization an allocation
may imply).  It keeps its split partials in a fixed array inside libfg.so
instead of a caller workspace.

Checked through the C ABI against fg_decode_attention, the entry point with
a caller-provided workspace, on two calls in a row with different queries
and lengths (the array keeps the previous call's contents), on a cache with
few (sequence, head) pairs so the split path and its scratch are in use.
Both entry points run the same kernels with the same split count in the
same order, so their outputs must be bit-identical; both are also checked
against the oracle's attention over the same cache contents.  This file
sorts last so a failure here cannot hide an earlier one."""
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


def test_noalloc_matches_workspace_entry_point_on_two_calls(fg):
    b, H, d, length, cap = 2, 4, 128, 300, 320
    h1 = H * d
    kv = fg.KVCache(b, H, d, cap, True, torch.float16, "cuda")
    ocache = olayer.KVCache(b, H, d, cap, True, "f16")
    assert fg.fg_decode_attention_workspace_bytes(kv) > 0          # the split path runs
    k = synth.normal((length, b, h1), 31, 1.3, torch.float16, "cuda")
    v = synth.normal((length, b, h1), 32, 1.3, torch.float16, "cuda")
    for p in range(length):
        fg.fg_kv_append(kv, k[p].contiguous(), v[p].contiguous(), p)
    ocache.store(k.cpu().numpy().astype(np.float64).transpose(1, 0, 2),
                 v.cpu().numpy().astype(np.float64).transpose(1, 0, 2), 0)
    for call, (pos, seed) in enumerate([(length - 1, 33), (length - 51, 34)]):
        q = synth.normal((b, h1), seed, 1.3, torch.float16, "cuda")
        ref = torch.empty_like(q)
        fg.fg_decode_attention(kv, q, pos, ref)
        got = torch.full_like(q, float("nan"))        # an unwritten output stays NaN and fails
        fg.fg_decode_attention_noalloc(kv, q, pos, got)
        fg.fg_sync_status()
        assert torch.equal(got, ref), f"call {call}: outputs differ from the workspace entry point"
        want = olayer.attention(q.cpu().numpy().astype(np.float64).reshape(b, 1, H, d),
                                ocache.k_val[:, :, :pos + 1], ocache.v_val[:, :, :pos + 1],
                                np.array([pos])).reshape(b, h1)
        err = np.max(np.abs(got.cpu().numpy().astype(np.float64) - want)) / np.max(np.abs(want))
        assert err <= 5e-3, f"call {call}: rel err {err} against the oracle"
