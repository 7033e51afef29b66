"""OPT-style transformer layer (prefill, and decode with KV Concat) in fp64 numpy.

Source: FlexGen notes (papercache.org, "FlexGen: High-Throughput Generative
Inference of Large Language Models with a Single GPU"), section
"背景知识 (Background)", the generative-inference equations:

  prefill, layer i, x in R^{b x s x h1}:
      x_K = x w_K ;  x_V = x w_V ;  x_Q = x w_Q
      x_Out = Softmax(x_Q x_K^T / sqrt(h1)) x_V w_O + x
      x^{i+1} = relu(x_Out w_1) w_2 + x_Out
  decode, layer i, t in R^{b x 1 x h1}:
      x_K <- Concat(x_K, t w_K) ;  x_V <- Concat(x_V, t w_V)
      t_Q = t w_Q
      t_Out = Softmax(t_Q x_K^T / sqrt(h1)) x_V w_O + t
      t^{i+1} = relu(t_Out w_1) w_2 + t_Out

and section "5. 近似方法": weights and the KV cache are stored in the 4-bit
group format and converted back to FP16 before compute.

Readings:
  * the prefill softmax is causal (generation; it also makes a decode step
    equal to the last row of a prefill over the extended sequence);
  * with H heads the score scale is 1/sqrt(h1/H) per head; H = 1 is the
    page's form 1/sqrt(h1);
  * the attention always reads K and V through the codec, including the
    tokens written in the same call; the new K/V rows are first rounded to
    the activation storage type (fp16, or fp32 for the fp32 configuration)
    and then quantized, so the integer codes are decided on the same values
    a GPU stores;
  * weights are dequantized to the activation type; all other arithmetic is
    fp64 with no intermediate rounding;
  * decode step t = 1..n writes cache slot s + t - 1 (0-based) and attends
    over slots 0..s + t - 1.

Matrix products and exp use numpy (fp64); there is no blocking, fusion or
reordering beyond the equations.  Test infrastructure only.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import codec


def _act_np(act_dtype: str):
    return {"f16": np.float16, "f32": np.float32}[act_dtype]


def weight_for_compute(w: np.ndarray, quantized: bool, act_dtype: str,
                       rows_per_chunk: int = 64) -> np.ndarray:
    """w: [K=in][N=out] in the storage type of the generated weights.
    Returns the matrix the layer multiplies by, in fp64: the raw weights,
    or dequant(quant(w)) grouped along the output channel (the last axis)
    and converted to the activation type.  Rows are processed in chunks only
    to bound the size of temporaries."""
    if not quantized:
        return np.asarray(w).astype(np.float64)
    out = np.empty(w.shape, dtype=np.float64)
    for r0 in range(0, w.shape[0], rows_per_chunk):
        blk = np.asarray(w[r0:r0 + rows_per_chunk])
        c, m, s = codec.quantize_g64(blk)
        out[r0:r0 + rows_per_chunk] = codec.dequant_g64(c, m, s, _act_np(act_dtype))
    return out


def dequant_weight(codes: np.ndarray, mins: np.ndarray, scales: np.ndarray, act_dtype: str,
                   rows_per_chunk: int = 64) -> np.ndarray:
    """A stored 4-bit weight ([K][N/2] codes, [K][N/64] mins and scales)
    converted back to the activation type, as fp64 (row chunks only bound
    the temporaries)."""
    K = codes.shape[0]
    out = np.empty((K, codes.shape[1] * 2), dtype=np.float64)
    for r0 in range(0, K, rows_per_chunk):
        sl = slice(r0, r0 + rows_per_chunk)
        out[sl] = codec.dequant_g64(codes[sl], mins[sl], scales[sl], _act_np(act_dtype))
    return out


@dataclass
class Weights:
    """Layer weights as the layer multiplies by them (fp64), x . w layout."""
    wq: np.ndarray
    wk: np.ndarray
    wv: np.ndarray
    wo: np.ndarray
    w1: np.ndarray
    w2: np.ndarray

    @staticmethod
    def prepare(raw: dict, quantized: bool, act_dtype: str) -> "Weights":
        return Weights(**{k: weight_for_compute(raw[k], quantized, act_dtype)
                          for k in ("wq", "wk", "wv", "wo", "w1", "w2")})


@dataclass
class KVCache:
    """One layer's cache, [b][H][capacity][d].  With the codec on it holds the
    codes and per-group (min, scale) exactly as stored, plus the fp64 values
    attention reads (dequantized to the activation type)."""
    b: int
    heads: int
    head_dim: int
    capacity: int
    quantized: bool
    act_dtype: str
    k_val: np.ndarray = field(init=False)
    v_val: np.ndarray = field(init=False)
    k_codes: np.ndarray | None = field(init=False, default=None)
    v_codes: np.ndarray | None = field(init=False, default=None)
    k_mins: np.ndarray | None = field(init=False, default=None)
    k_scales: np.ndarray | None = field(init=False, default=None)
    v_mins: np.ndarray | None = field(init=False, default=None)
    v_scales: np.ndarray | None = field(init=False, default=None)

    def __post_init__(self):
        shp = (self.b, self.heads, self.capacity, self.head_dim)
        self.k_val = np.zeros(shp)
        self.v_val = np.zeros(shp)
        if self.quantized:
            cshp = shp[:-1] + (self.head_dim // 2,)
            mshp = shp[:-1] + (self.head_dim // codec.GROUP,)
            self.k_codes = np.zeros(cshp, np.uint8)
            self.v_codes = np.zeros(cshp, np.uint8)
            self.k_mins = np.zeros(mshp, np.float32)
            self.k_scales = np.zeros(mshp, np.float32)
            self.v_mins = np.zeros(mshp, np.float32)
            self.v_scales = np.zeros(mshp, np.float32)

    def store(self, k: np.ndarray, v: np.ndarray, pos0: int) -> None:
        """Concat: write rows k, v ([b][T][h1], fp64) at slots pos0..pos0+T-1.
        Each row is rounded to the activation type; with the codec on it is
        quantized in groups of 64 along the hidden dimension."""
        b, T, h1 = k.shape
        assert h1 == self.heads * self.head_dim and pos0 + T <= self.capacity
        sl = slice(pos0, pos0 + T)
        for name, rows in (("k", k), ("v", v)):
            act = rows.astype(_act_np(self.act_dtype))
            act = act.reshape(b, T, self.heads, self.head_dim).transpose(0, 2, 1, 3)
            if self.quantized:
                c, m, s = codec.quantize_g64(np.ascontiguousarray(act))
                getattr(self, name + "_codes")[:, :, sl] = c
                getattr(self, name + "_mins")[:, :, sl] = m
                getattr(self, name + "_scales")[:, :, sl] = s
                val = codec.dequant_g64(c, m, s, _act_np(self.act_dtype))
            else:
                val = act
            getattr(self, name + "_val")[:, :, sl] = val.astype(np.float64)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos: np.ndarray) -> np.ndarray:
    """Causal multi-head attention.
    q: [b][Tq][H][d]; k, v: [b][H][Tk][d]; q_pos: absolute slot of each query.
    Key j is visible to a query at slot p iff j <= p.  Scale 1/sqrt(d)."""
    d = q.shape[-1]
    scores = np.einsum("bqhd,bhkd->bhqk", q, k) / np.sqrt(d)
    tk = k.shape[2]
    visible = np.arange(tk)[None, :] <= np.asarray(q_pos)[:, None]   # [Tq][Tk]
    scores = np.where(visible[None, None], scores, -np.inf)
    mx = scores.max(axis=-1, keepdims=True)
    p = np.exp(scores - mx)
    p = p / p.sum(axis=-1, keepdims=True)
    return np.einsum("bhqk,bhkd->bqhd", p, v)



def topk_keep(tokens: int, percent: int = 10) -> int:
    """How many tokens the sparse approximation keeps: the top `percent` per
    cent of `tokens`, rounded up, and at least one ("5. 近似方法", sparse
    attention: the top 10% of the value cache).  Integer arithmetic, so that
    e.g. 530 tokens keep 53, not the 54 a float ceil(0.1 * 530) gives."""
    assert tokens >= 1 and 1 <= percent <= 100
    return max(1, (tokens * percent + 99) // 100)


def attention_topk(q: np.ndarray, k: np.ndarray, v: np.ndarray, keep: int):
    """Top-K sparse decode attention ("5. 近似方法", sparse attention).

    q: [b][H][d], one query per (sequence, head) at the newest slot;
    k, v: [b][H][T][d], every one of the T cached tokens visible.
    The page's steps, in its order:
      1. the attention matrix: p = Softmax(q k^T / sqrt(d)) over all T tokens;
      2. for each query, the indices of its `keep` largest entries (Top-K);
      3. the other tokens are dropped, and only the selected rows of V are
         read: out = sum over the selected i of p_i v_i.
    Readings: the kept weights are the ones step 1 computed over all tokens
    (the page drops tokens after the attention matrix exists, and says
    nothing of renormalising); among equal scores the lower token index
    ranks first; keep >= T keeps every token (dense attention).
    Returns (out [b][H][d], idx [b][H][min(keep, T)] ascending)."""
    b, H, T, d = k.shape
    kk = min(keep, T)
    scores = np.einsum("bhd,bhtd->bht", q, k) / np.sqrt(d)
    mx = scores.max(axis=-1, keepdims=True)
    p = np.exp(scores - mx)
    p = p / p.sum(axis=-1, keepdims=True)
    out = np.zeros((b, H, d))
    idx = np.zeros((b, H, kk), np.int64)
    for bi in range(b):
        for h in range(H):
            # descending score, ties by ascending index (lexsort: last key is primary)
            order = np.lexsort((np.arange(T), -scores[bi, h]))
            sel = np.sort(order[:kk])
            idx[bi, h] = sel
            out[bi, h] = p[bi, h, sel] @ v[bi, h, sel]
    return out, idx

def _relu(a: np.ndarray) -> np.ndarray:
    return np.maximum(a, 0.0)


def prefill_layer(x: np.ndarray, w: Weights, cache: KVCache) -> np.ndarray:
    """x: [b][s][h1] (fp64 values of the stored activations).  Writes slots
    0..s-1 of the cache and returns x^{i+1} in fp64."""
    b, s, h1 = x.shape
    H, d = cache.heads, cache.head_dim
    xk = x @ w.wk
    xv = x @ w.wv
    xq = x @ w.wq
    cache.store(xk, xv, 0)
    att = attention(xq.reshape(b, s, H, d), cache.k_val[:, :, :s], cache.v_val[:, :, :s],
                    np.arange(s))
    x_out = att.reshape(b, s, h1) @ w.wo + x
    return _relu(x_out @ w.w1) @ w.w2 + x_out


def decode_layer(t: np.ndarray, w: Weights, cache: KVCache, pos: int) -> np.ndarray:
    """t: [b][h1].  Appends t w_K, t w_V at slot pos, attends over 0..pos and
    returns t^{i+1} in fp64."""
    b, h1 = t.shape
    H, d = cache.heads, cache.head_dim
    tk = t @ w.wk
    tv = t @ w.wv
    cache.store(tk[:, None], tv[:, None], pos)
    tq = t @ w.wq
    att = attention(tq.reshape(b, 1, H, d), cache.k_val[:, :, :pos + 1],
                    cache.v_val[:, :, :pos + 1], np.array([pos]))
    t_out = att.reshape(b, h1) @ w.wo + t
    return _relu(t_out @ w.w1) @ w.w2 + t_out


def run_block(x0: np.ndarray, t_inputs: np.ndarray, layers: list[Weights], heads: int,
              quantized: bool, act_dtype: str):
    """One zig-zag block: the prompt through every layer, then n decode steps,
    each through every layer.  x0: [b][s][h1]; t_inputs: [n][b][h1] (the
    embedding fed to layer 0 at each step).  Returns (prefill output of the
    last layer, list of per-step outputs of the last layer, caches)."""
    b, s, h1 = x0.shape
    n = t_inputs.shape[0]
    caches = [KVCache(b, heads, h1 // heads, s + n, quantized, act_dtype) for _ in layers]
    x = np.asarray(x0, dtype=np.float64)
    for w, c in zip(layers, caches):
        x = prefill_layer(x, w, c)
    outs = []
    for t_idx in range(n):
        t = np.asarray(t_inputs[t_idx], dtype=np.float64)
        for w, c in zip(layers, caches):
            t = decode_layer(t, w, c, s + t_idx)
        outs.append(t)
    return x, outs, caches
