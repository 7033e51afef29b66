#!/usr/bin/env python
"""Decode throughput of the int4 group-64 OPT layer stack on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config opt-6.7b]
                    [--impl ours|reference]

One step is one zig-zag block of the FlexGen notes ("4. 卸载策略"): the
b-sequence prompt (s tokens) through all l layers, then n decode steps, each
through all l layers, with weights and KV cache in 4-bit groups of 64
("5. 近似方法").  Inputs are seeded synthetic tensors of the OPT shapes
(weights N(0, 0.02), prompt and per-step embeddings N(0, 1)); everything is
resident in HBM before the timed region.  The reported value is decode
tokens/s: b*n*K (times the number of ranks) over the device time of the
decode phases of the K timed steps (max over ranks).

With --impl reference the CPU oracle (the plain fp64/fp32 restatement of the
page, under oracle/) is timed on the host cores on a bounded sample of the
same workload and printed in the same format.

Multi-GPU (torchrun): replicas only; every rank runs its own block (its own
prompt seeds, the same weights) with no collective on the data path; the
timing is the max over ranks and the value sums all ranks' tokens.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "decode tokens/s (OPT-6.7B shape, int4 W+KV); achieved HBM GB/s vs ~8 TB/s"
Q4 = 0.5 + 8.0 / 64.0   # bytes per element: 4-bit code + fp32 (min, scale) per 64
# bytes per weight of each decode-copy format (fg_pack_weight): the default
# carries the stored fp32 pairs, the opt-in one fp16 pairs
PACK_BYTES = {0: Q4, 1: 0.5 + 4.0 / 64.0}


# DRAM traffic of the dominant decode kernel class from one ncu capture
# (profiles/gemm_q4ts_qkv_opt-6.7b_b64.md): dram__bytes_read.sum +
# dram__bytes_write.sum of x.[w_Q w_K w_V] (M = 64, K = 4096, N = 12288),
# averaged over 4 launches, beside that launch's algorithmic bytes (weights as
# stored + X read + Y written).  Valid only for the kernel sources it was
# taken on (their hash); scaled to the class's average launch by algorithmic
# bytes (the products differ only in size, and the capture reads each weight
# byte once).
TRAFFIC = {"gemm_q4_decode": {
    "sources": ("int4_group_quantized_gb300/csrc/gemm_q4ts.cu", "int4_group_quantized_gb300/csrc/q4_convert.cuh",
                "int4_group_quantized_gb300/csrc/q4_dev.cuh", "int4_group_quantized_gb300/csrc/tc_ptx.cuh"),
    "sha256_16": ("3157f5bfb3e916e3", "bdc48444633d6cb6", "360d7c9967f0a780", "396e7d83852eb72d"),
    "dram_bytes": 32036096.0,
    "algorithmic_bytes": 4096 * 12288 * Q4 + 2 * 64 * (4096 + 3 * 4096),
    "capture": "ncu, x.[w_Q w_K w_V] M=64 K=4096 N=12288, one launch (K splits reduced in the cluster)"}}


def traffic_per_launch(kernel: str, algorithmic_per_launch: float):
    """Measured DRAM bytes per launch of `kernel`, scaled from its capture,
    or None when the capture does not match the current sources."""
    import hashlib
    t = TRAFFIC.get(kernel)
    if t is None:
        return None
    for path, want in zip(t["sources"], t["sha256_16"]):
        try:
            got = hashlib.sha256(open(os.path.join(ROOT, path), "rb").read()).hexdigest()[:16]
        except OSError:
            return None
        if got != want:
            return None
    return t["dram_bytes"] / t["algorithmic_bytes"] * algorithmic_per_launch


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "tflops": d["bf16_tflops"],
                "tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "tflops": 1900.0, "tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.rows = []
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            ident = str(device)
        self.cmd = ["nvidia-smi", "-i", ident, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "200"]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in self.rows:
            try:
                sm.append(float(r[0]))
                mx = float(r[1])
            except ValueError:
                continue
            for nm, v in zip(names, r[3:]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------
# algorithmic work (FlexGen notes "背景知识" memory formulas, "附录 A.3" compute terms)
# ---------------------------------------------------------------------------------------

def decode_product_bytes(w, b, pack_format: int = 0) -> float:
    """One decode step of one layer, all four products: every 4-bit weight
    once for the whole block, in the form the decode products read it (the
    decode copy, PACK_BYTES per weight), plus the fp16 activations they read
    and write: t in and Q|K|V out; attention output and residual t in, t_Out
    out; t_Out in, hidden out; hidden and residual t_Out in, t^{i+1} out."""
    h1, h2 = w.h1, w.h2
    weights = (4 * h1 * h1 + 2 * h1 * h2) * PACK_BYTES[pack_format]
    act = 2 * b * ((h1 + 3 * h1) + (h1 + h1 + h1) + (h1 + h2) + (h2 + h1 + h1))
    return weights + act


def decode_product_flops(w, b) -> float:
    return 2.0 * b * (4 * w.h1 * w.h1 + 2 * w.h1 * w.h2)


def decode_attn_bytes(w, b, length) -> float:
    """The append and attention launch: read K and V of `length` tokens
    (4-bit, the new one included), write the appended K/V row once, read q
    and the new K/V rows (fp16), write the output (fp16)."""
    return 2 * b * w.h1 * length * Q4 + 2 * b * w.h1 * Q4 + 2 * b * w.h1 * 4


def topk_attn_bytes(w, length, keep) -> float:
    """Top-K sparse attention alone (nothing appended): every K row of
    `length` tokens, `keep` V rows per (sequence, head), q and the output
    (fp16)."""
    return w.b * w.h1 * length * Q4 + w.b * w.heads * min(keep, length) * w.head_dim * Q4 + 2 * w.b * w.h1 * 2


def prefill_product_flops(w, b, s) -> float:
    return 2.0 * b * s * (4 * w.h1 * w.h1 + 2 * w.h1 * w.h2)


def prefill_attn_flops(w, b, s) -> float:
    return 4.0 * b * w.h1 * (s * (s + 1) / 2)


def decode_step_bytes(w, b, length, pack_format: int = 0) -> float:
    return decode_product_bytes(w, b, pack_format) + decode_attn_bytes(w, b, length)


# ---------------------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline)
# ---------------------------------------------------------------------------------------

def oracle_decode_sample(w, budget_s: float = 20.0) -> dict:
    """Times the oracle on one decode step of one layer for the whole block at
    cache length s + n/2, including the dequantization of that layer's 4-bit
    weights (stored quantized, converted back before compute).  Returns
    decode tokens/s of the full l-layer model on this host."""
    from oracle import codec as ocodec
    from oracle import layer as olayer

    raw = synth.layer_weights(w, 0, "cpu")
    stored = {}
    for m in synth.MATS:     # model preparation, not timed
        a = raw[m].numpy()
        parts = [ocodec.quantize_g64(a[r:r + 64]) for r in range(0, a.shape[0], 64)]
        stored[m] = tuple(np.concatenate([p[i] for p in parts]) for i in range(3))
    length = w.s + w.n // 2
    cache = olayer.KVCache(w.b, w.heads, w.head_dim, length + 1, True, w.act)
    rng = np.random.default_rng(0)
    cache.k_val[:, :, :length] = rng.standard_normal((w.b, w.heads, length, w.head_dim))
    cache.v_val[:, :, :length] = rng.standard_normal((w.b, w.heads, length, w.head_dim))
    t_in = synth.decode_inputs(w, n=1, device="cpu")[0].numpy().astype(np.float64)
    act = np.float16 if w.act == "f16" else np.float32
    times = []
    t_start = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        wts = olayer.Weights(**{m: olayer.dequant_weight(*stored[m], w.act) for m in synth.MATS})
        olayer.decode_layer(t_in, wts, cache, length)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > budget_s or len(times) >= 3:
            break
    t = statistics.median(times)
    return {"value": w.b / (t * w.l), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "threads": os.environ.get("OMP_NUM_THREADS") or os.environ.get("OPENBLAS_NUM_THREADS") or "blas default",
            "sample": (f"one decode step of one {w.name} layer for all b={w.b} sequences at cache length "
                       f"{length}, weight dequantization included, median of {len(times)}; scaled to "
                       f"l={w.l} layers"),
            "seconds_per_layer_step": t, "samples": len(times)}


# ---------------------------------------------------------------------------------------
# replicas (torchrun): every rank runs its own block, no collective on the data path
# ---------------------------------------------------------------------------------------

def max_over_ranks(values, world: int, device) -> list:
    """Per-rank seconds -> their element-wise max over the ranks: the job's
    clock is its slowest replica."""
    if world <= 1:
        return list(values)
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def job_tokens(w, steps: int, world: int) -> int:
    """Decode tokens the whole job produces: b*n per step on every rank."""
    return w.b * w.n * steps * world


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    res = oracle_decode_sample(w)
    line = {"impl": "reference", "metric": METRIC, "value": res["value"], "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            # not run end to end: the oracle's time for one sampled layer-step,
            # scaled to the l layers and n decode steps of one bench step
            "ms_per_step": res["seconds_per_layer_step"] * w.l * w.n * 1e3,
            "ms_per_step_kind": "scaled from the sample: seconds_per_layer_step * l * n",
            "sampled_work": {"layer_steps": res["samples"], "seconds_per_layer_step": res["seconds_per_layer_step"],
                             "b": w.b, "cache_length": w.s + w.n // 2},
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "l": w.l, "h1": w.h1, "h2": w.h2, "heads": w.heads, "b": w.b,
                       "s": w.s, "n": w.n},
            "cpu_baseline": {k: res[k] for k in ("value", "unit", "cores", "kind", "sample", "threads")},
            "e2e": {"value": res["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------------------

def run_ours(args, w, rank, world, device):
    import int4_group_quantized_gb300 as fg

    dt = synth.torch_dtype(w.act)
    torch.cuda.set_device(device)
    dev = torch.device("cuda", device)
    st = torch.cuda.current_stream()

    # model preparation (not timed): fp16 weights drawn on the device one layer
    # at a time, quantized by the library's codec kernel, fp16 copy freed
    layers, kvs = [], []
    qbytes, qtime = 0, 0.0
    for i in range(w.l):
        raw = synth.layer_weights(w, i, dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        L = fg.Layer.from_dense(raw, w.heads, quantized=True)
        e1.record()
        e1.synchronize()
        qtime += e0.elapsed_time(e1) / 1e3
        qbytes += sum(t.numel() for t in raw.values()) * (2 + Q4)
        layers.append(L)
        del raw
        kvs.append(fg.KVCache(w.b, w.heads, w.head_dim, w.s + w.n, True, dt, dev))
    blk = fg.Block(layers, kvs)
    ws = fg.workspace(max(fg.fg_prefill_block_workspace_bytes(layers[0], w.b, w.s),
                          fg.fg_decode_block_workspace_bytes(layers[0], w.b, w.s + w.n)), dev)
    x = synth.prompt(w, device=dev, seed_offset=rank)
    tin = synth.decode_inputs(w, device=dev, seed_offset=rank)
    y = torch.empty_like(x)
    outs = torch.empty_like(tin)

    # decode steps replay CUDA graphs recorded by the first warm-up step
    # (fg_decode_block_step_graphed); the profiled pass below runs them directly
    graphs = None if args.no_graph else fg.GraphCache()

    def decode_step(t_in, pos, out):
        if graphs is not None and not args._prof:
            fg.fg_decode_block_step_graphed(graphs, blk, t_in, pos, out, ws, st)
        else:
            fg.fg_decode_block_step(blk, t_in, pos, out, ws, st)

    def step(evs=None):
        if evs:
            evs[0].record(st)
        fg.fg_profile_phase(0) if args._prof else None
        fg.fg_prefill_block(blk, x, y, ws, st)
        if evs:
            evs[1].record(st)
        fg.fg_profile_phase(1) if args._prof else None
        for t in range(w.n):
            decode_step(tin[t], w.s + t, outs[t])
        if evs:
            evs[2].record(st)

    args._prof = False
    for _ in range(args.warmup):
        step()
    fg.fg_sync_status(st)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    n0 = fg.fg_launch_count()
    with ClockSampler(device) as clk:
        t_wall = time.perf_counter()
        for k in range(args.steps):
            step(evs[k])
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    n_launch = fg.fg_launch_count() - n0
    fg.fg_sync_status(st)

    # per-kernel device times: the same K steps again with an event pair
    # around every library launch (kept out of the timed region above)
    launches_per_step = w.l * 16 + w.n * w.l * 16
    fg.fg_profile_start(args.steps * launches_per_step + 64)
    args._prof = True
    for k in range(args.steps):
        step()
    torch.cuda.synchronize()
    prof = fg.fg_profile_stop()
    args._prof = False
    pre_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[1].elapsed_time(e[2]) for e in evs]
    tot_ms = [e[0].elapsed_time(e[2]) for e in evs]
    dec_total = sum(dec_ms) / 1e3
    tot_total = sum(tot_ms) / 1e3
    pre_total = sum(pre_ms) / 1e3
    dec_total, tot_total, pre_total = max_over_ranks([dec_total, tot_total, pre_total], world, dev)
    nonfinite = int((~torch.isfinite(outs)).sum().item())

    # end to end through the public API with host buffers: the prompt comes from
    # pinned host memory before the decode phase (outside the timed region, like
    # the prefill); inside it, each step's embedding is copied in from pinned
    # host memory and each step's output copied back
    x_h = x.cpu().pin_memory()
    tin_h = tin.cpu().pin_memory()
    out_h = torch.empty(outs.shape, dtype=outs.dtype, pin_memory=True)
    x_d = torch.empty_like(x)
    t_d = torch.empty_like(tin[0])
    e2e_ms = []
    h2d_step = d2h_step = 0
    for k in range(args.steps + 1):   # the first pass records the graphs of these buffers, untimed
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        x_d.copy_(x_h, non_blocking=True)
        fg.fg_prefill_block(blk, x_d, y, ws, st)
        e[0].record(st)
        h2d_step = d2h_step = 0
        for t in range(w.n):
            t_d.copy_(tin_h[t], non_blocking=True)
            h2d_step += t_d.numel() * t_d.element_size()
            decode_step(t_d, w.s + t, outs[t])
            out_h[t].copy_(outs[t], non_blocking=True)
            d2h_step += outs[t].numel() * outs[t].element_size()
        e[1].record(st)
        torch.cuda.synchronize()
        if k > 0:
            e2e_ms.append(e[0].elapsed_time(e[1]))
    e2e_dec = max_over_ranks([sum(e2e_ms) / 1e3], world, dev)[0]

    # the same decode layer-steps on finite data: one layer of the stack, its
    # cache filled by its own prefill of a fresh N(0, 1) prompt, and a fresh
    # N(0, 1) input at every step (the chained stack above overflows fp16 after
    # a few layers: the page's layer has no normalisation); per-kernel device
    # time per layer-step, beside the chained run's
    finite, topk = finite_layer_steps(fg, w, layers[w.l // 2], dev, st, args.steps)
    offload = None if args.no_offload else offload_timing(fg, w, layers, kvs, tin, ws, dev, st)

    if rank != 0:
        return
    pk = peaks()
    K = args.steps
    tokens = job_tokens(w, K, world)
    value = tokens / dec_total
    # roofline of the decode phase's dominant kernel class
    mean_len = statistics.mean(w.s + t + 1 for t in range(w.n))
    dec_prof = prof.get(1, {})
    pre_prof = prof.get(0, {})
    work = {}
    for name, (cnt, ms) in dec_prof.items():
        if name.startswith("gemm"):
            flops = decode_product_flops(w, w.b) * w.l * w.n * K
            byts = decode_product_bytes(w, w.b) * w.l * w.n * K
            # split-K reduction launches belong to the products they finish
            work[name] = (byts, flops, ms, cnt)
        elif name == "attn_decode":
            work[name] = (decode_attn_bytes(w, w.b, mean_len) * w.l * w.n * K, 4.0 * w.b * w.h1 * mean_len * w.l * w.n * K, ms, cnt)
    dom = max(dec_prof.items(), key=lambda kv: kv[1][1])[0] if dec_prof else None
    roof = None
    if dom in work:
        byts, flops, ms, cnt = work[dom]
        if dom.startswith("gemm") and w.b >= 128:
            ach = flops / (ms / 1e3) / 1e12
            roof = {"bound": "tensor", "achieved": ach, "peak": pk["tflops_sustained"], "unit": "TFLOP/s",
                    "frac": ach / pk["tflops_sustained"], "traffic": None, "kernel": dom}
        else:
            ach = byts / (ms / 1e3) / 1e9
            roof = {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": ach / pk["hbm_gbs"], "traffic": None, "kernel": dom}
        roof.update({"launches": cnt, "avg_launch_us": ms / cnt * 1e3,
                     "algorithmic_per_launch": (byts if roof["unit"] == "GB/s" else flops) / cnt,
                     "peak_source": pk["source"] + (" sustained" if roof["unit"] == "TFLOP/s" else "")})
        if roof["unit"] == "GB/s":
            tr = traffic_per_launch(dom, byts / cnt)
            roof["traffic"] = tr
            roof["traffic_source"] = TRAFFIC[dom]["capture"] + ", scaled by algorithmic bytes" if tr else None
    roof_pre = None
    g_pre = {k: v for k, v in pre_prof.items() if k.startswith("gemm")}
    if g_pre:
        ms = sum(v[1] for v in g_pre.values())
        cnt = sum(v[0] for v in g_pre.values())
        ach = prefill_product_flops(w, w.b, w.s) * w.l * K / (ms / 1e3) / 1e12
        # the products alternate with attention inside the prefill, and the SM
        # clock stays at its maximum there: the burst figure is the fair peak
        roof_pre = {"bound": "tensor", "achieved": ach, "peak": pk["tflops"], "unit": "TFLOP/s",
                    "frac": ach / pk["tflops"], "traffic": None, "kernel": "+".join(sorted(g_pre)),
                    "launches": cnt, "avg_launch_us": ms / cnt * 1e3,
                    "peak_source": pk["source"] + " burst (fp16 and bf16 share the dense rate)",
                    "frac_of_sustained": ach / pk["tflops_sustained"]}
    dec_bytes = sum(decode_step_bytes(w, w.b, w.s + t + 1) for t in range(w.n)) * w.l * K * world
    cpu = oracle_decode_sample(w, budget_s=args.cpu_budget) if not args.no_cpu else None
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": tot_total / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": w.name, "l": w.l, "h1": w.h1, "h2": w.h2, "heads": w.heads, "b": w.b,
                   "s": w.s, "n": w.n, "weights": "int4 g64 (fp32 min/scale)", "kv": "int4 g64",
                   "l2": "inputs larger than L2 (%.1f GB of 4-bit weights + %.1f GB of 4-bit KV)" % (
                       sum(L.nbytes() for L in layers) / 1e9, sum(c.nbytes() for c in kvs) / 1e9),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "value_definition": "b*n*steps*ranks / decode-phase device time (max over ranks)"},
        "roofline": roof, "roofline_prefill": roof_pre,
        "decode_achieved_gbs_step": dec_bytes / dec_total / 1e9,
        "prefill_tok_s": w.b * w.s * K * world / pre_total,
        "generation_tok_s": w.b * w.n * K * world / tot_total,
        "decode_ms_per_step": dec_total / K * 1e3, "prefill_ms_per_step": pre_total / K * 1e3,
        "quantize_gbs": qbytes / qtime / 1e9 if qtime else None,
        "kernels": {f"{'prefill' if p == 0 else 'decode'}:{k}": {"launches": v[0], "ms": round(v[1], 3)}
                    for p, d in prof.items() for k, v in d.items()},
        "gpu_launches": int(n_launch), "nonfinite_decode_outputs": nonfinite,
        "decode_path": "direct calls" if args.no_graph else "fg_decode_block_step_graphed (CUDA graph per step)",
        "cpu_baseline": cpu and {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample", "threads")},
        "e2e": {"value": w.b * w.n * K * world / e2e_dec, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d_step, "d2h_bytes_per_step": d2h_step,
                "definition": ("decode phase through fg_decode_block_step with every step's embedding copied in "
                               "from pinned host memory and its output copied back, inside the timed region; "
                               "the prompt copy and the prefill run before it")},
        "finite_data_check": {
            "chained_us_per_layer_step": {k.split(":", 1)[1]: round(v[1] / (w.l * w.n * K) * 1e3, 2)
                                          for k, v in ((f"decode:{a}", b) for a, b in dec_prof.items())},
            "finite_us_per_layer_step": finite},
        "topk_attention_4bit_s": topk,
        "offload_c2c": offload,
        "clocks": clocks, "wall_s_timed": t_wall,
    }
    print(json.dumps(line), flush=True)


def finite_layer_steps(fg, w, L, dev, st, steps: int) -> dict:
    """Per-kernel device microseconds per decode layer-step of one layer on
    finite data (see run_ours)."""
    dt = synth.torch_dtype(w.act)
    kv = fg.KVCache(w.b, w.heads, w.head_dim, w.s + w.n, True, dt, dev)
    x = synth.prompt(w, device=dev, seed_offset=101)
    y = torch.empty_like(x)
    ws = fg.workspace(max(fg.fg_prefill_workspace_bytes(L, w.b, w.s),
                          fg.fg_decode_workspace_bytes(L, w.b, w.s + w.n)), dev)
    tin = synth.decode_inputs(w, device=dev, seed_offset=102)
    out = torch.empty_like(tin[0])
    total = {}
    for k in range(max(1, steps)):
        fg.fg_prefill_layer(L, x, kv, y, ws, st)
        torch.cuda.synchronize()
        fg.fg_profile_start(w.n * 16 + 64)
        fg.fg_profile_phase(1)
        for t in range(w.n):
            fg.fg_decode_step(L, tin[t], w.s + t, kv, out, ws, st)
        torch.cuda.synchronize()
        prof = fg.fg_profile_stop().get(1, {})
        assert torch.isfinite(out).all(), "finite-data decode produced a non-finite output"
        for name, (cnt, ms) in prof.items():
            total[name] = total.get(name, 0.0) + ms
    per_step = {name: round(ms / (w.n * max(1, steps)) * 1e3, 2) for name, ms in total.items()}
    return per_step, topk_attention_timing(fg, w, kv, dev, st)


def offload_timing(fg, w, layers, kvs, tin, ws, dev, st, steps: int = 4) -> dict:
    """Decode steps with every layer's decode copies in pinned host memory,
    streamed over NVLink-C2C into a two-half device stage while the previous
    layer computes (fg_decode_block_step_offload, Algorithm 1's overlap):
    device time per step and the host-to-device rate it implies.  Runs on the
    stack's caches after the timed region (it rewrites slots s..s+steps-1)."""
    host = [L.offloaded(stored_too=False) for L in layers]
    blk = fg.Block(host, kvs)
    stage = fg.workspace(fg.fg_offload_stage_bytes(layers[0]), dev)
    copy = torch.cuda.Stream(device=dev)
    out = torch.empty_like(tin[0])
    for t in range(2):   # warm-up
        fg.fg_decode_block_step_offload(blk, tin[t], w.s + t, out, ws, stage, st, copy)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for t in range(steps):
        fg.fg_decode_block_step_offload(blk, tin[t], w.s + t, out, ws, stage, st, copy)
    e1.record(st)
    e1.synchronize()
    fg.fg_sync_status()
    ms = e0.elapsed_time(e1) / steps
    per_step = w.l * fg.fg_offload_stage_bytes(layers[0]) / 2
    res = {"steps": steps, "ms_per_step": round(ms, 3), "tokens_per_s": round(w.b / (ms * 1e-3), 1),
           "h2d_bytes_per_step": per_step, "h2d_gbs": round(per_step / (ms * 1e-3) / 1e9, 1),
           "definition": "decode copies of all layers in pinned host memory, copied layer by layer on a "
                         "second stream while the previous layer computes; KV cache and activations in HBM"}
    # the same weights read in place by the decode kernels' bulk copies over
    # NVLink-C2C (no stage), where the pinned pages are mapped at the same
    # address on the device
    if all(_device_maps_host_at_same_address(L.w[m].packed.data_ptr()) for L in host for m in fg.Layer.MATS):
        blk0 = fg.Block(host, kvs)
        fg.fg_decode_block_step(blk0, tin[0], w.s, out, ws, st)
        torch.cuda.synchronize()
        e0.record(st)
        for t in range(steps):
            fg.fg_decode_block_step(blk0, tin[t], w.s + t, out, ws, st)
        e1.record(st)
        e1.synchronize()
        fg.fg_sync_status()
        zms = e0.elapsed_time(e1) / steps
        res["in_place"] = {"ms_per_step": round(zms, 3), "tokens_per_s": round(w.b / (zms * 1e-3), 1),
                           "host_read_gbs": round(per_step / (zms * 1e-3) / 1e9, 1)}
    return res


def _device_maps_host_at_same_address(ptr: int) -> bool:
    """cudaPointerGetAttributes: pinned host memory whose device address is
    the host address (so a kernel may read it through the pointer)."""
    import ctypes

    class Attr(ctypes.Structure):   # cudaPointerAttributes as the CUDA 13 runtime header declares it
        _fields_ = [("type", ctypes.c_int), ("device", ctypes.c_int), ("devicePointer", ctypes.c_void_p),
                    ("hostPointer", ctypes.c_void_p), ("reserved", ctypes.c_long * 8)]
    for name in ("libcudart.so", "libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            rt = None
    if rt is None:
        return False
    a = Attr()
    if rt.cudaPointerGetAttributes(ctypes.byref(a), ctypes.c_void_p(ptr)) != 0:
        return False
    return a.type == 1 and a.devicePointer == ptr and a.hostPointer == ptr


def topk_attention_timing(fg, w, kv, dev, st, calls: int = 10) -> dict:
    """Top-K sparse attention (the page's 4-bit-S setting, the top 10% of the
    tokens) over a full finite cache of s + n tokens: device time per call,
    L2 flushed before each call (the cache's K alone is below L2's size)."""
    length = w.s + w.n
    keep = fg.topk_keep(length)
    q = synth.normal((w.b, w.h1), 5, 1.0, synth.torch_dtype(w.act), dev)
    out = torch.empty_like(q)
    flush = torch.empty(3 * 129 * 2 ** 20 // 4, dtype=torch.float32, device=dev)
    ms = []
    with torch.cuda.stream(st):
        for k in range(calls + 3):
            flush.fill_(float(k))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            fg.fg_decode_attention_topk(kv, q, length - 1, keep, out, stream=st)
            e1.record(st)
            e1.synchronize()
            if k >= 3:
                ms.append(e0.elapsed_time(e1))
    fg.fg_sync_status()
    us = statistics.mean(ms) * 1e3
    byts = topk_attn_bytes(w, length, keep)
    return {"tokens": length, "keep": keep, "us_per_call": round(us, 2), "algorithmic_bytes": byts,
            "achieved_gbs": round(byts / (us * 1e-6) / 1e9, 1),
            "dense_bytes_same_cache": 2 * w.b * w.h1 * length * Q4 + 2 * w.b * w.h1 * 2}


CASES = ("linear-qkv", "linear-o", "linear-fc1", "linear-fc2", "prefill-linear-fc1", "attn-decode",
         "attn-decode-topk", "prefill-layer")


def run_case(args, w, device):
    """One kernel class at the workload's shapes, with a small device
    footprint (one layer): the command the ncu summaries under profiles/ are
    taken with.  Enough weight copies (or caches) rotate that the inputs of
    consecutive calls exceed L2; the calls are captured once in a CUDA graph
    and the graph is replayed `--steps` times after `--warmup` replays, so the
    printed time per call is device time without host launch overhead."""
    import int4_group_quantized_gb300 as fg
    torch.cuda.set_device(device)
    dev = torch.device("cuda", device)
    dt = synth.torch_dtype(w.act)
    name = args.case
    l2 = 3 * 129 * 2 ** 20
    if name.startswith("linear") or name.startswith("prefill-linear"):
        mat = {"qkv": "wq", "o": "wo", "fc1": "w1", "fc2": "w2"}[name.split("-")[-1]]
        K, N = synth.weight_shape(w, mat)
        if mat == "wq":
            N *= 3
        prefill = name.startswith("prefill")
        M = min(w.b * w.s, 8192) if prefill else (args.m or w.b)   # a few GB at most on the device
        per = K * N * (2 if prefill else Q4)
        copies = 1 if prefill else max(2, min(32, int(-(-l2 // per))))
        Ws = []
        for c in range(copies):
            w16 = synth.normal((K, N), 7 + c, synth.WEIGHT_STD, dt, dev)
            Ws.append(fg.QuantWeight.from_dense(w16, not prefill))
            del w16
        x = synth.normal((M, K), 8, 1.0, dt, dev)
        y = torch.empty((M, N), dtype=dt, device=dev)
        ws = fg.workspace(max(fg.fg_linear_workspace_bytes(M, K, N, not prefill, dt), 1), dev)
        calls = [lambda W=W: fg.fg_linear(W, x, y, ws=ws) for W in Ws]
        shape = {"M": M, "K": K, "N": N, "copies": copies}
        if not prefill:   # weights once (0.625 B each) + x in and y out (fp16)
            shape["algorithmic_bytes"] = K * N * Q4 + 2 * M * (K + N)
    else:
        L = fg.Layer.from_dense(synth.layer_weights(w, 0, dev), w.heads, True)
        x = synth.prompt(w, device=dev)
        y = torch.empty_like(x)
        ws = fg.workspace(max(fg.fg_prefill_workspace_bytes(L, w.b, w.s),
                              fg.fg_decode_workspace_bytes(L, w.b, w.s + w.n)), dev)
        if name.startswith("attn-decode"):
            kv_bytes = 2 * w.b * w.h1 * (w.s + w.n) * 0.625
            kvs = [fg.KVCache(w.b, w.heads, w.head_dim, w.s + w.n, True, dt, dev)
                   for _ in range(max(2, int(-(-l2 // kv_bytes))))]
            for kv in kvs:
                fg.fg_prefill_layer(L, x, kv, y, ws)       # fills slots 0..s-1
            q = synth.normal((w.b, w.h1), 9, 1.0, dt, dev)
            out = torch.empty_like(q)
            pos = w.s + w.n // 2
            if name == "attn-decode-topk":
                keep = fg.topk_keep(pos + 1)
                calls = [lambda kv=kv: fg.fg_decode_attention_topk(kv, q, pos, keep, out) for kv in kvs]
                algo = topk_attn_bytes(w, pos + 1, keep)
            else:
                calls = [lambda kv=kv: fg.fg_decode_attention(kv, q, pos, out) for kv in kvs]
                algo = 2 * w.b * w.h1 * (pos + 1) * Q4 + 2 * w.b * w.h1 * 2   # K, V; q and the output
        else:
            kv = fg.KVCache(w.b, w.heads, w.head_dim, w.s + w.n, True, dt, dev)
            calls = [lambda: fg.fg_prefill_layer(L, x, kv, y, ws)]
        shape = {"b": w.b, "s": w.s, "h1": w.h1, "heads": w.heads, "copies": len(calls)}
        if name.startswith("attn-decode"):
            shape.update({"len": pos + 1, "algorithmic_bytes": algo})
            if name == "attn-decode-topk":
                shape["keep"] = keep
    reps = max(1, 16 // len(calls)) * len(calls) if len(calls) < 16 else len(calls)
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        for k in range(reps):
            calls[k % len(calls)]()
        torch.cuda.synchronize()
        graph.capture_begin()
        for k in range(reps):
            calls[k % len(calls)]()
        graph.capture_end()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        graph.replay()
    e1.record()
    e1.synchronize()
    fg.fg_sync_status()
    us = e0.elapsed_time(e1) / (args.steps * reps) * 1e3
    rec = {"case": name, "workload": w.name, "shape": shape, "calls_per_replay": reps, "us_per_call": us}
    if "algorithmic_bytes" in shape:
        rec["achieved_gbs"] = shape["algorithmic_bytes"] / (us * 1e-6) / 1e9
    print(json.dumps(rec), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="opt-6.7b", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle timing")
    ap.add_argument("--no-graph", action="store_true", help="decode steps by direct calls, not replayed graphs")
    ap.add_argument("--no-offload", action="store_true", help="skip the host-offloaded decode timing")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--m", type=int, default=None, help="rows of a decode-product case (default: the block size)")
    ap.add_argument("--case", choices=CASES, default=None,
                    help="time one kernel class at the workload's shapes (for profilers)")
    args = ap.parse_args()
    w = synth.WORKLOADS[args.config]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    if args.case:
        run_case(args, w, local)
        return
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    run_ours(args, w, rank, world, local)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
