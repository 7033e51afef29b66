"""Seeded synthetic inputs and workload shapes, shared by tests, bench and smoke.

This module holds no arithmetic of the method: it only draws normal random
tensors with fixed seeds and lists the workload shapes.  Both the CUDA path
and the oracle take their inputs from here.

Workloads follow the FlexGen notes' OPT shapes (prompt s = 512, n = 32
generated tokens; "背景知识" and "实验结果" sections), plus a one-layer
exact-formula check.  Weights are N(0, 0.02), prompts and decode-step
embeddings N(0, 1); there is no tokenizer, embedding table or LM head on
the page, so every decode step feeds a fresh N(0, 1) embedding to layer 0.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    cfg_id: int
    l: int
    h1: int
    h2: int
    heads: int
    b: int
    s: int
    n: int
    act: str          # "f16" or "f32"

    @property
    def head_dim(self) -> int:
        return self.h1 // self.heads


WORKLOADS = {
    "tiny": Workload("tiny", 0, 1, 64, 256, 1, 2, 8, 4, "f32"),
    "opt-125m": Workload("opt-125m", 1, 12, 768, 3072, 12, 32, 512, 32, "f16"),
    "opt-6.7b": Workload("opt-6.7b", 2, 32, 4096, 16384, 32, 64, 512, 32, "f16"),
    "opt-30b": Workload("opt-30b", 3, 48, 7168, 28672, 56, 256, 512, 32, "f16"),
    "opt-175b": Workload("opt-175b", 4, 96, 12288, 49152, 96, 64, 512, 32, "f16"),
}

MATS = ("wq", "wk", "wv", "wo", "w1", "w2")
WEIGHT_STD = 0.02


def torch_dtype(act: str) -> torch.dtype:
    return {"f16": torch.float16, "f32": torch.float32}[act]


def normal(shape, seed: int, std: float = 1.0, dtype=torch.float16, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32 from a generator seeded with `seed` on
    `device`, then cast to `dtype`.  CPU and CUDA generators give different
    streams; tests hand the oracle copies of whatever was drawn."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def weight_seed(cfg_id: int, layer: int, mat_id: int) -> int:
    return 1_000_003 * cfg_id + 16 * layer + mat_id


def weight_shape(w: Workload, mat: str) -> tuple[int, int]:
    """[K = in][N = out], so the layer computes x . w."""
    return {"wq": (w.h1, w.h1), "wk": (w.h1, w.h1), "wv": (w.h1, w.h1),
            "wo": (w.h1, w.h1), "w1": (w.h1, w.h2), "w2": (w.h2, w.h1)}[mat]


def layer_weights(w: Workload, layer: int, device="cpu", dtype=None) -> dict:
    dt = torch_dtype(w.act) if dtype is None else dtype
    return {m: normal(weight_shape(w, m), weight_seed(w.cfg_id, layer, i), WEIGHT_STD, dt, device)
            for i, m in enumerate(MATS)}


def prompt(w: Workload, b: int | None = None, s: int | None = None, device="cpu", seed_offset: int = 0):
    b = w.b if b is None else b
    s = w.s if s is None else s
    return normal((b, s, w.h1), 1_000_003 * w.cfg_id + 900_000 + seed_offset, 1.0,
                  torch_dtype(w.act), device)


def decode_inputs(w: Workload, b: int | None = None, n: int | None = None, device="cpu",
                  seed_offset: int = 0):
    b = w.b if b is None else b
    n = w.n if n is None else n
    return normal((n, b, w.h1), 1_000_003 * w.cfg_id + 950_000 + seed_offset, 1.0,
                  torch_dtype(w.act), device)
