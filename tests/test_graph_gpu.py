"""fg_decode_block_step_graphed: the zig-zag block's decode step recorded
once into a CUDA graph and replayed (FlexGen notes, "4. 卸载策略": the same
layer loop at every decode step).  The replayed steps must give exactly the
bits of the direct calls, count the same launches, and keep one graph per
distinct step."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fg():
    import int4_group_quantized_gb300 as fg
    return fg


def _block(fg, w, nl):
    raw = [synth.layer_weights(w, i, "cuda") for i in range(nl)]
    layers = [fg.Layer.from_dense(r, w.heads, quantized=True) for r in raw]
    dt = synth.torch_dtype(w.act)
    kvs = [fg.KVCache(w.b, w.heads, w.head_dim, w.s + w.n, True, dt, "cuda") for _ in layers]
    blk = fg.Block(layers, kvs)
    ws = fg.workspace(max(fg.fg_prefill_block_workspace_bytes(layers[0], w.b, w.s),
                          fg.fg_decode_block_workspace_bytes(layers[0], w.b, w.s + w.n)), "cuda")
    return blk, ws


@pytest.mark.parametrize("name,nl,n", [("opt-125m", 3, 6), ("small16", 2, 5)])
def test_graphed_steps_equal_direct_steps(fg, name, nl, n):
    w = synth.WORKLOADS[name] if name in synth.WORKLOADS else synth.Workload(name, 9, 2, 256, 512, 2, 5, 77, 6, "f16")
    blk, ws = _block(fg, w, nl)
    x = synth.prompt(w, device="cuda")
    tin = synth.decode_inputs(w, device="cuda")[:n]
    y = torch.empty_like(x)
    direct = torch.empty_like(tin)
    fg.fg_prefill_block(blk, x, y, ws)
    for t in range(n):
        fg.fg_decode_block_step(blk, tin[t], w.s + t, direct[t], ws)
    fg.fg_sync_status()
    cache = fg.GraphCache()
    graphed = torch.empty_like(tin)
    for rep in range(3):          # record on the first pass, replay on the next two
        graphed.fill_(float("nan"))
        fg.fg_prefill_block(blk, x, y, ws)
        n0 = fg.fg_launch_count()
        for t in range(n):
            fg.fg_decode_block_step_graphed(cache, blk, tin[t], w.s + t, graphed[t], ws)
        fg.fg_sync_status()
        launches = fg.fg_launch_count() - n0
        assert torch.equal(graphed, direct), f"pass {rep}: outputs differ from the direct steps"
        if rep == 0:
            first = launches
        else:
            assert launches == first, (launches, first)
        assert len(cache) == n
    cache.close()


def test_graphed_step_errors_match_direct(fg):
    w = synth.WORKLOADS["opt-125m"]
    blk, ws = _block(fg, w, 1)
    cache = fg.GraphCache()
    t = torch.zeros((w.b, w.h1), dtype=torch.float16, device="cuda")
    y = torch.empty_like(t)
    with pytest.raises(fg.FGError) as e:
        fg.fg_decode_block_step_graphed(cache, blk, t, w.s + w.n, y, ws)   # pos at capacity
    assert e.value.status == 4
    assert len(cache) == 0
