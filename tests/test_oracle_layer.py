"""CPU pins for the oracle's layer math (FlexGen notes, "背景知识" generative
inference equations) and the page's byte/flop formulas.

Pins: the page's printed OPT-175B memory figures, element counts of the
oracle's own tensors, brute-force attention with explicit loops, PyTorch's
fp64 scaled_dot_product_attention as a textbook layer, the identity special
case, and decode == last row of a causal prefill over the extended sequence.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import codec, formulas, layer

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "flexgen_memory.txt")


def _golden():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            out[k] = float(v)
    return out


def test_page_memory_figures():
    g = _golden()
    l, h1, h2 = int(g["l"]), int(g["h1"]), int(g["h2"])
    w = formulas.weight_bytes_fp16(l, h1, h2)
    assert w == 347_892_350_976
    assert abs(w / 2 ** 30 - g["weights_GB"]) / g["weights_GB"] < 0.005     # 324.0 GiB vs "325 GB"
    kv = formulas.kv_bytes_fp16_peak(int(g["kv_b"]), l, h1, int(g["kv_s"]), int(g["kv_n"]))
    assert kv == 1_314_259_992_576
    assert abs(kv / 2 ** 40 - g["kv_TB"]) / g["kv_TB"] < 0.005             # 1.195 TiB vs "1.2 TB"
    assert round(kv / w, 1) == g["kv_over_weights"]                         # 3.78 vs "3.8x"


def test_formulas_match_tensor_element_counts():
    h1, h2, b, s, n, H = 128, 512, 3, 5, 4, 2
    shapes = {"wq": (h1, h1), "wk": (h1, h1), "wv": (h1, h1), "wo": (h1, h1), "w1": (h1, h2), "w2": (h2, h1)}
    assert sum(2 * a * c for a, c in shapes.values()) == formulas.weight_bytes_fp16(1, h1, h2)
    cache = layer.KVCache(b, H, h1 // H, s + n, False, "f16")
    assert 2 * (cache.k_val.size + cache.v_val.size) == formulas.kv_bytes_fp16_peak(b, 1, h1, s, n)
    qc = layer.KVCache(b, H, h1 // H, s + n, True, "f16")
    q4 = qc.k_codes.nbytes + qc.v_codes.nbytes + qc.k_mins.nbytes * 4
    assert q4 == formulas.q4_bytes(2 * b * h1 * (s + n))
    # flops: 2 per multiply-add of each product the prefill equations write
    mm = 2 * b * s * (4 * h1 * h1 + 2 * h1 * h2)
    att = 2 * (2 * b * s * s * h1)
    assert formulas.prefill_flops_layer(b, s, h1, h2) == mm + att
    # mean KV bytes over the n steps equals the mean of the per-step lengths s + t, t = 0..n
    mean_len = np.mean([s + t for t in range(n + 1)])
    assert formulas.kv_bytes_fp16_mean_layer(b, s, n, h1) == 4 * b * mean_len * h1


def _tiny_weights(h1, h2, seed, quantized, act="f32"):
    rng = np.random.default_rng(seed)
    dt = np.float32 if act == "f32" else np.float16
    raw = {k: (rng.standard_normal(shp) * 0.05).astype(dt) for k, shp in
           {"wq": (h1, h1), "wk": (h1, h1), "wv": (h1, h1), "wo": (h1, h1),
            "w1": (h1, h2), "w2": (h2, h1)}.items()}
    return raw, layer.Weights.prepare(raw, quantized, act)


def test_attention_matches_explicit_loops():
    rng = np.random.default_rng(0)
    b, s, H, d = 2, 7, 2, 64
    q = rng.standard_normal((b, s, H, d))
    k = rng.standard_normal((b, H, s, d))
    v = rng.standard_normal((b, H, s, d))
    got = layer.attention(q, k, v, np.arange(s))
    for bi in range(b):
        for h in range(H):
            for i in range(s):
                sc = [sum(q[bi, i, h, e] * k[bi, h, j, e] for e in range(d)) / math.sqrt(d) for j in range(i + 1)]
                m = max(sc)
                w = [math.exp(x - m) for x in sc]
                z = sum(w)
                for e in range(d):
                    ref = sum(w[j] * v[bi, h, j, e] for j in range(i + 1)) / z
                    assert abs(got[bi, i, h, e] - ref) < 1e-12


def _textbook_prefill(x, raw, H):
    """Unquantized layer with torch fp64 and scaled_dot_product_attention; K/V
    rounded to fp32 like the stored cache."""
    X = torch.from_numpy(x)
    W = {k: torch.from_numpy(np.asarray(v, dtype=np.float64)) for k, v in raw.items()}
    b, s, h1 = X.shape
    d = h1 // H
    q = (X @ W["wq"]).view(b, s, H, d).transpose(1, 2)
    k = (X @ W["wk"]).float().double().view(b, s, H, d).transpose(1, 2)
    v = (X @ W["wv"]).float().double().view(b, s, H, d).transpose(1, 2)
    a = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    a = a.transpose(1, 2).reshape(b, s, h1)
    xo = a @ W["wo"] + X
    return (torch.relu(xo @ W["w1"]) @ W["w2"] + xo).numpy()


@pytest.mark.parametrize("H", [1, 2])
def test_unquantized_prefill_equals_textbook(H):
    h1, h2, b, s = 128, 256, 2, 9
    raw, w = _tiny_weights(h1, h2, 1, quantized=False)
    x = np.random.default_rng(2).standard_normal((b, s, h1)).astype(np.float32).astype(np.float64)
    cache = layer.KVCache(b, H, h1 // H, s, False, "f32")
    got = layer.prefill_layer(x, w, cache)
    ref = _textbook_prefill(x, raw, H)
    assert np.max(np.abs(got - ref)) < 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_zero_output_weights_give_identity():
    h1, h2, b, s = 64, 256, 2, 5
    raw, _ = _tiny_weights(h1, h2, 3, quantized=False)
    raw["wo"][:] = 0
    raw["w2"][:] = 0
    for quant in (False, True):
        w = layer.Weights.prepare(raw, quant, "f32")
        x = np.random.default_rng(4).standard_normal((b, s, h1))
        cache = layer.KVCache(b, 1, h1, s + 1, quant, "f32")
        assert np.array_equal(layer.prefill_layer(x, w, cache), x)
        t = np.random.default_rng(5).standard_normal((b, h1))
        assert np.array_equal(layer.decode_layer(t, w, cache, s), t)


@pytest.mark.parametrize("quant", [False, True])
def test_single_token_prefill_equals_decode_into_empty_cache(quant):
    h1, h2, b, H = 128, 256, 3, 2
    _, w = _tiny_weights(h1, h2, 6, quant)
    t = np.random.default_rng(7).standard_normal((b, h1)).astype(np.float32).astype(np.float64)
    c1 = layer.KVCache(b, H, h1 // H, 4, quant, "f32")
    c2 = layer.KVCache(b, H, h1 // H, 4, quant, "f32")
    y1 = layer.prefill_layer(t[:, None, :], w, c1)[:, 0]
    y2 = layer.decode_layer(t, w, c2, 0)
    assert np.max(np.abs(y1 - y2)) < 1e-12
    if quant:
        assert np.array_equal(c1.k_codes, c2.k_codes) and np.array_equal(c1.v_scales, c2.v_scales)


@pytest.mark.parametrize("quant,act", [(False, "f32"), (True, "f32"), (True, "f16")])
def test_decode_equals_last_row_of_extended_prefill(quant, act):
    """Decode at slot s+t-1 equals row s+t-1 of a causal prefill over the
    prompt extended with the t decode inputs, for a 2-layer stack."""
    h1, h2, b, s, n, H = 128, 256, 2, 6, 3, 2
    dt = np.float32 if act == "f32" else np.float16
    layers = [_tiny_weights(h1, h2, 10 + i, quant, act)[1] for i in range(2)]
    rng = np.random.default_rng(11)
    x0 = rng.standard_normal((b, s, h1)).astype(dt).astype(np.float64)
    tin = rng.standard_normal((n, b, h1)).astype(dt).astype(np.float64)
    _, outs, caches = layer.run_block(x0, tin, layers, H, quant, act)
    ext = np.concatenate([x0, tin.transpose(1, 0, 2)], axis=1)
    full, _, caches_full = layer.run_block(ext, np.zeros((0, b, h1)), layers, H, quant, act)
    for t in range(n):
        assert np.max(np.abs(outs[t] - full[:, s + t])) < 1e-12 * max(1.0, np.abs(full).max())
    if quant:
        for c, cf in zip(caches, caches_full):
            assert np.array_equal(c.k_codes, cf.k_codes) and np.array_equal(c.v_codes, cf.v_codes)


def test_quantized_kv_is_grouped_along_hidden_per_token():
    h1, H, b = 256, 2, 2
    rng = np.random.default_rng(12)
    k = rng.standard_normal((b, 3, h1))
    v = rng.standard_normal((b, 3, h1))
    c = layer.KVCache(b, H, h1 // H, 3, True, "f16")
    c.store(k, v, 0)
    # token 1 of sequence 1, head 1, hidden 128..255 == two groups of 64 of that row
    row = k[1, 1, 128:].astype(np.float16)
    codes, mins, scales = codec.quantize_g64(row[None])
    assert np.array_equal(c.k_codes[1, 1, 1], codes[0])
    assert np.array_equal(c.k_mins[1, 1, 1], mins[0])


def test_weights_grouped_along_output_channel():
    raw = np.random.default_rng(13).standard_normal((3, 128)).astype(np.float16)
    w = layer.weight_for_compute(raw, True, "f16")
    # row k (fixed input index) holds two groups: outputs 0..63 and 64..127
    for k in range(3):
        for g in range(2):
            seg = raw[k, 64 * g:64 * g + 64].astype(np.float64)
            rt = w[k, 64 * g:64 * g + 64]
            step = (seg.max() - seg.min()) / 15
            assert np.max(np.abs(seg - rt)) <= step / 2 + 1e-3


# ---- the remaining formulas, each against the sizes of the oracle's own tensors --------

def _small():
    return dict(h1=128, h2=512, b=3, H=2, s=5, n=4, l=2)


def test_activation_bytes_is_one_fp16_hidden_state():
    c = _small()
    bls = c["b"] * c["s"]
    x = np.zeros((c["b"], c["s"], c["h1"]), np.float16)
    assert formulas.activation_bytes_fp16(bls, c["h1"]) == x.nbytes


def test_zigzag_peak_mem_is_weights_plus_activation_plus_kv():
    """Appendix A.2's zig-zag peak: the fp16 weights of all l layers, one fp16
    hidden state of the block, and the fp16 KV cache of every layer grown to
    s + n tokens -- summed from the oracle's own tensors."""
    c = _small()
    h1, h2, b, s, n, l, H = c["h1"], c["h2"], c["b"], c["s"], c["n"], c["l"], c["H"]
    raws = [_tiny_weights(h1, h2, 40 + i, False, "f16")[0] for i in range(l)]
    w_bytes = sum(a.nbytes for r in raws for a in r.values())
    act = np.zeros((b, h1), np.float16).nbytes
    caches = [layer.KVCache(b, H, h1 // H, s + n, False, "f16") for _ in range(l)]
    kv = sum(2 * (cc.k_val.size + cc.v_val.size) for cc in caches)   # fp16 storage: 2 bytes a value
    assert formulas.zigzag_peak_mem(w_bytes, h1, b, l, s, n) == w_bytes + act + kv


def test_causal_prefill_flops_count_the_visible_pairs():
    c = _small()
    h1, h2, b = c["h1"], c["h2"], c["b"]
    for s in (1, 2, 7, 64):
        visible = int(np.sum(np.arange(s)[None, :] <= np.arange(s)[:, None]))
        dense = formulas.prefill_flops_layer(b, s, h1, h2)
        causal = formulas.prefill_flops_layer(b, s, h1, h2, causal=True)
        # 2 products (scores and values) x 2 flops per multiply-add x h1 per pair
        assert dense - causal == 4 * b * h1 * (s * s - visible)
        if s == 1:
            assert dense == causal


def test_decode_flops_are_the_decode_layer_products():
    """2 flops per multiply-add of every product decode_layer performs, from
    the shapes of the oracle's weights and cache."""
    c = _small()
    h1, h2, b, H, length = c["h1"], c["h2"], c["b"], c["H"], 9
    raw, w = _tiny_weights(h1, h2, 41, True, "f16")
    macs = sum(b * m.shape[0] * m.shape[1] for m in (w.wq, w.wk, w.wv, w.wo, w.w1, w.w2))
    cache = layer.KVCache(b, H, h1 // H, length, True, "f16")
    d = cache.head_dim
    macs += 2 * b * H * length * d          # q . K^T over `length` slots, then p . V
    assert formulas.decode_flops_layer(b, h1, h2, length) == 2 * macs


def test_decode_bytes_are_the_tensors_a_step_touches():
    """Stored 4-bit weights, the KV slots read and the one written, and the
    fp16 activations of one decode step, from the oracle's own arrays."""
    c = _small()
    h1, h2, b, H, length = c["h1"], c["h2"], c["b"], c["H"], 9
    raw, _ = _tiny_weights(h1, h2, 42, False, "f16")
    wbytes = 0
    for m in raw.values():
        cd, mn, sc = codec.quantize_g64(m)
        wbytes += cd.nbytes + mn.nbytes + sc.nbytes
    cache = layer.KVCache(b, H, h1 // H, length, True, "f16")
    arrs = (cache.k_codes, cache.v_codes, cache.k_mins, cache.k_scales, cache.v_mins, cache.v_scales)
    kv_read = sum(a[:, :, :length].nbytes for a in arrs)
    kv_write = sum(a[:, :, :1].nbytes for a in arrs)
    f16 = lambda *shape: np.zeros(shape, np.float16).nbytes
    act = (f16(b, h1) + f16(b, 3 * h1)                      # t in, Q|K|V out
           + f16(b, h1) * 3 + f16(b, h1)                    # q, new K, new V in; attention out
           + f16(b, h1) * 2 + f16(b, h1)                    # attention out, residual t in; t_Out out
           + f16(b, h1) + f16(b, h2)                        # t_Out in, hidden out
           + f16(b, h2) + f16(b, h1) + f16(b, h1))          # hidden, residual t_Out in; t^{i+1} out
    assert formulas.decode_bytes_layer_q4(b, h1, h2, length) == wbytes + kv_read + kv_write + act


def test_generation_throughput_counts_block_tokens():
    """b n / t: the tokens run_block generates (one per sequence per step)
    over the time."""
    h1, h2, H = 64, 128, 1
    raw, w = _tiny_weights(h1, h2, 43, False)
    rng = np.random.default_rng(44)
    b, s, n = 3, 4, 5
    _, outs, _ = layer.run_block(rng.standard_normal((b, s, h1)), rng.standard_normal((n, b, h1)), [w], H,
                                 False, "f32")
    tokens = sum(o.shape[0] for o in outs)
    assert formulas.generation_throughput(b, n, 2.5) == tokens / 2.5


def test_bench_byte_counts_equal_the_oracle_formula():
    """bench.py's roofline numerator (its own restatement, since the timed
    path may not import the oracle) equals the oracle's formula; with the
    fp16-metadata decode copy it differs by exactly the weights' smaller
    pairs."""
    import bench
    import synth
    for name in ("opt-125m", "opt-6.7b", "opt-30b", "opt-175b"):
        w = synth.WORKLOADS[name]
        for length in (w.s + 1, w.s + w.n):
            want = formulas.decode_bytes_layer_q4(w.b, w.h1, w.h2, length)
            assert bench.decode_step_bytes(w, w.b, length, 0) == pytest.approx(want, rel=1e-12)
            diff = formulas.layer_weight_elems(w.h1, w.h2) * (8.0 - 4.0) / 64.0
            assert bench.decode_step_bytes(w, w.b, length, 1) == pytest.approx(want - diff, rel=1e-12)
        assert bench.decode_product_flops(w, w.b) + 4.0 * w.b * w.h1 * (w.s + 1) == \
            formulas.decode_flops_layer(w.b, w.h1, w.h2, w.s + 1)
