"""Byte and flop counts the FlexGen notes print, written out (test oracle).

Source: FlexGen notes (papercache.org, "FlexGen: High-Throughput Generative
Inference of Large Language Models with a Single GPU"):
  * "背景知识", memory-bottleneck paragraph: fp16 parameter bytes
    l (8 h1^2 + 4 h1 h2); peak KV bytes 4 b l h1 (s + n); throughput b n / t;
  * "4. 卸载策略", cost-model paragraph: per-layer fp16 weight bytes
    8 h1^2 + 4 h1 h2, activation bytes 2 bls h1, mean KV bytes
    4 bls (s + n/2) h1;
  * "附录 A.2": zig-zag peak memory w + 2 h1 bls + 4 h1 bls l (s + n);
  * "附录 A.3": prefill compute bls (8 s h1^2 + 4 s h1 h2) matmul flops plus
    4 bls s^2 h1 batched-matmul flops; decode attention 4 bls (s + n/2) h1.

The 4-bit storage used here adds one fp32 (min, scale) pair per 64 codes:
0.5 + 8/64 = 0.625 bytes per element (format reading, not from the page).
Test infrastructure only.
"""
from __future__ import annotations

Q4_BYTES_PER_ELEM = 0.5 + 8.0 / 64.0


def weight_bytes_fp16(l: int, h1: int, h2: int) -> int:
    return l * (8 * h1 * h1 + 4 * h1 * h2)


def kv_bytes_fp16_peak(b: int, l: int, h1: int, s: int, n: int) -> int:
    return 4 * b * l * h1 * (s + n)


def layer_weight_elems(h1: int, h2: int) -> int:
    return 4 * h1 * h1 + 2 * h1 * h2


def activation_bytes_fp16(bls: int, h1: int) -> int:
    return 2 * bls * h1


def kv_bytes_fp16_mean_layer(bls: int, s: int, n: int, h1: int) -> float:
    return 4 * bls * (s + n / 2) * h1


def zigzag_peak_mem(w_bytes: float, h1: int, bls: int, l: int, s: int, n: int) -> float:
    return w_bytes + 2 * h1 * bls + 4 * h1 * bls * l * (s + n)


def prefill_flops_layer(bls: int, s: int, h1: int, h2: int, causal: bool = False) -> float:
    """Matmul flops plus attention flops of one layer's prefill; the page's
    attention term 4 bls s^2 h1 counts the dense s x s score and value
    products; causal=True counts the lower triangle (s(s+1)/2 pairs)."""
    mm = bls * (8 * s * h1 * h1 + 4 * s * h1 * h2)
    att = 4 * bls * s * s * h1 if not causal else 4 * bls * (s * (s + 1) // 2) * h1
    return mm + att


def decode_flops_layer(bls: int, h1: int, h2: int, length: int) -> float:
    """One decode step of one layer: 2 flops per weight per sequence, plus
    4 h1 flops per cached token per sequence (scores and values)."""
    return bls * (2 * layer_weight_elems(h1, h2) + 4 * h1 * length)


def q4_bytes(elems: float) -> float:
    return elems * Q4_BYTES_PER_ELEM


def decode_bytes_layer_q4(bls: int, h1: int, h2: int, length: int) -> float:
    """Algorithmic HBM bytes of one decode step of one layer with 4-bit
    weights and KV: every weight once (zig-zag reuse across the block),
    the K and V cache of `length` tokens (including the appended one), the
    appended K/V row written once, and fp16 activations in and out of each
    of the five products."""
    w = q4_bytes(layer_weight_elems(h1, h2))
    kv_read = q4_bytes(2 * bls * h1 * length)
    kv_write = q4_bytes(2 * bls * h1)
    act = 2 * bls * (h1 + 3 * h1 + h1 + h1 + h1 + h1 + h2 + h2 + h1)
    return w + kv_read + kv_write + act


def generation_throughput(b: int, n: int, t_seconds: float) -> float:
    return b * n / t_seconds
