"""fg_decode_block_step_offload: Algorithm 1 of the FlexGen notes ("4. 卸载策略":
load the next layer's weights while computing this one) with the weights in
host memory, streamed over NVLink-C2C into a two-half device stage.  The
same kernels read the same bytes, so the outputs must be bit-identical to
the resident block step, with the copy stream apart from the compute
stream or the same."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fg():
    import int4_group_quantized_gb300 as fg
    return fg


@pytest.mark.parametrize("name,nl,n", [("opt-125m", 4, 5), ("opt-6.7b", 3, 3)])
@pytest.mark.parametrize("same_stream", [False, True])
def test_offloaded_steps_equal_resident_steps(fg, name, nl, n, same_stream):
    w = synth.WORKLOADS[name]
    raw = [synth.layer_weights(w, i, "cuda") for i in range(nl)]
    layers = [fg.Layer.from_dense(r, w.heads, quantized=True) for r in raw]
    del raw
    dt = synth.torch_dtype(w.act)
    kv_a = [fg.KVCache(w.b, w.heads, w.head_dim, w.s + w.n, True, dt, "cuda") for _ in layers]
    kv_b = [fg.KVCache(w.b, w.heads, w.head_dim, w.s + w.n, True, dt, "cuda") for _ in layers]
    resident = fg.Block(layers, kv_a)
    host_layers = [L.offloaded() for L in layers]
    offl = fg.Block(host_layers, kv_b)
    assert host_layers[0].w["wq"].packed.device.type == "cpu"
    ws = fg.workspace(max(fg.fg_prefill_block_workspace_bytes(layers[0], w.b, w.s),
                          fg.fg_decode_block_workspace_bytes(layers[0], w.b, w.s + w.n)), "cuda")
    stage = fg.workspace(fg.fg_offload_stage_bytes(layers[0]), "cuda")
    x = synth.prompt(w, device="cuda")
    tin = synth.decode_inputs(w, device="cuda")[:n]
    y = torch.empty_like(x)
    fg.fg_prefill_block(resident, x, y, ws)
    fg.fg_prefill_block(fg.Block(layers, kv_b), x, y, ws)   # the same prompt into the second cache
    copy = torch.cuda.current_stream() if same_stream else torch.cuda.Stream()
    want = torch.empty_like(tin)
    got = torch.full_like(tin, float("nan"))
    for t in range(n):
        fg.fg_decode_block_step(resident, tin[t], w.s + t, want[t], ws)
        fg.fg_decode_block_step_offload(offl, tin[t], w.s + t, got[t], ws, stage, copy_stream=copy)
    fg.fg_sync_status()
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    for a, b in zip(kv_a, kv_b):
        assert torch.equal(a.k_codes, b.k_codes) and torch.equal(a.v_codes, b.v_codes)
