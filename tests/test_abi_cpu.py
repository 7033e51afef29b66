"""CPU checks of the C ABI: libfg.so builds, loads, exports every function
include/fg.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fg():
    import __graft_entry__
    __graft_entry__.build()
    import int4_group_quantized_gb300 as fg
    return fg


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(fg_[a-z0-9_]+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(fg):
    names = _declared()
    assert {"fg_quantize_g64", "fg_dequant_g64", "fg_prefill_layer", "fg_decode_step",
            "fg_kv_append"} <= names
    for n in sorted(names):
        assert hasattr(fg.lib, n), n


def test_version_and_status_strings(fg):
    assert "sm_103a" in fg.fg_version()
    for code, name in fg.STATUS.items():
        assert fg.lib.fg_status_str(code).decode() == name


def test_codec_argument_errors(fg):
    L = fg.lib
    p = ctypes.c_void_p(16)
    assert L.fg_quantize_g64(p, 0, 2, 65, p, p, p, None) == 2          # FG_ERR_SHAPE
    assert b"multiple of 64" in L.fg_last_error()
    assert L.fg_quantize_g64(p, 7, 2, 64, p, p, p, None) == 1          # bad dtype
    assert L.fg_quantize_g64(None, 0, 2, 64, p, p, p, None) == 1       # null x
    assert L.fg_quantize_g64(ctypes.c_void_p(18), 0, 2, 64, p, p, p, None) == 3  # misaligned
    assert L.fg_quantize_g64(None, 0, 0, 64, None, None, None, None) == 0        # empty: no-op
    assert L.fg_dequant_g64(p, p, p, 1, 100, p, 0, None) == 2


def _layer(fg, h1=128, h2=256, heads=2, codec=1, dtype=0, packed=True):
    P = 4096
    wm = lambda K, N: fg.fg_wmat(P, P, P, P, K, N, P if packed else None, 0)
    return fg.fg_layer(wm(h1, h1), wm(h1, h1), wm(h1, h1), wm(h1, h1), wm(h1, h2), wm(h2, h1),
                       h1, h2, heads, codec, dtype)


def _kv(fg, b=2, cap=16, heads=2, d=64, codec=1, dtype=0):
    P = 4096
    return fg.fg_kv(P, P, P, P, P, P, P, P, b, cap, heads, d, codec, dtype)


def test_layer_argument_errors(fg):
    L = fg.lib
    lay, kv = _layer(fg), _kv(fg)
    P = ctypes.c_void_p(4096)
    ws = fg.lib.fg_decode_workspace_bytes(ctypes.byref(lay), 2, 16)
    assert ws > 0
    # pos at capacity
    assert L.fg_decode_step(ctypes.byref(lay), P, 2, 16, ctypes.byref(kv), P, P, ws, None) == 4
    assert L.fg_decode_step(ctypes.byref(lay), P, 2, -1, ctypes.byref(kv), P, P, ws, None) == 4
    # workspace too small
    assert L.fg_decode_step(ctypes.byref(lay), P, 2, 3, ctypes.byref(kv), P, P, ws - 1, None) == 5
    # b differs from the cache
    assert L.fg_decode_step(ctypes.byref(lay), P, 3, 3, ctypes.byref(kv), P, P, ws, None) == 2
    # head_dim 96 is not implemented
    bad = _layer(fg, h1=192, heads=2)
    assert L.fg_prefill_layer(ctypes.byref(bad), P, 2, 4, ctypes.byref(kv), P, P, ws, None) == 8
    # h2 not a multiple of 64
    bad = _layer(fg, h2=200)
    assert L.fg_prefill_layer(ctypes.byref(bad), P, 2, 4, ctypes.byref(kv), P, P, ws, None) == 2
    # wrong matrix shape
    bad = _layer(fg)
    bad.w1.N = 128
    assert L.fg_prefill_layer(ctypes.byref(bad), P, 2, 4, ctypes.byref(kv), P, P, ws, None) == 2
    # s beyond capacity
    assert L.fg_prefill_layer(ctypes.byref(lay), P, 2, 17, ctypes.byref(kv), P, P, 1 << 30, None) == 4
    # cache codec differs from layer codec
    kv2 = _kv(fg, codec=0)
    assert L.fg_prefill_layer(ctypes.byref(lay), P, 2, 4, ctypes.byref(kv2), P, P, 1 << 30, None) == 1
    # kv append outside capacity
    assert L.fg_kv_append(ctypes.byref(kv), P, P, 16, None) == 4
    # misaligned activation
    assert L.fg_decode_step(ctypes.byref(lay), ctypes.c_void_p(4098), 2, 3, ctypes.byref(kv), P, P, ws,
                            None) == 3
    # fp16 4-bit decode without the decode copy of every matrix
    bare = _layer(fg, packed=False)
    assert L.fg_decode_step(ctypes.byref(bare), P, 2, 3, ctypes.byref(kv), P, P, ws, None) == 1
    assert b"decode copy" in L.fg_last_error()
    assert L.fg_decode_workspace_bytes(ctypes.byref(bare), 2, 16) == 0
    # decode copies in two formats, or an unknown format
    mixed = _layer(fg)
    mixed.w1.packed_format = 1
    assert L.fg_decode_step(ctypes.byref(mixed), P, 2, 3, ctypes.byref(kv), P, P, ws, None) == 1
    mixed.w1.packed_format = 7
    assert L.fg_decode_step(ctypes.byref(mixed), P, 2, 3, ctypes.byref(kv), P, P, ws, None) == 1
    # fp32 layers need no decode copy
    f32 = _layer(fg, dtype=1, packed=False)
    assert fg.lib.fg_decode_workspace_bytes(ctypes.byref(f32), 2, 16) > 0


def test_pack_weight_sizes_and_errors(fg):
    L = fg.lib
    assert L.fg_pack_weight_bytes(4096, 12288, 0) == 4096 * 12288 * 5 // 8        # 0.625 B per weight
    assert L.fg_pack_weight_bytes(4096, 12288, 1) == 4096 * 12288 * 9 // 16       # 0.5625 B per weight
    assert L.fg_pack_weight_bytes(4096, 12288, 2) == 0
    assert L.fg_pack_weight_bytes(4096, 4160, 0) == 0                               # N % 128
    P = 4096
    w = fg.fg_wmat(P, P, P, None, 256, 512, None, 0)
    assert L.fg_pack_weight(ctypes.byref(w), 2, ctypes.c_void_p(P), None) == 1
    assert L.fg_pack_weight(ctypes.byref(w), 0, None, None) == 1
    w.N = 320
    assert L.fg_pack_weight(ctypes.byref(w), 0, ctypes.c_void_p(P), None) == 2


def test_noalloc_attention_host_errors(fg):
    """fg_decode_attention_noalloc rejects bad arguments on the host, before
    any CUDA call (these need no GPU)."""
    L = fg.lib
    P = ctypes.c_void_p(4096)
    assert L.fg_decode_attention_noalloc(None, P, 256, 3, P, 256, None) == 1           # FG_ERR_ARG
    bad = _kv(fg, heads=2, d=96)
    assert L.fg_decode_attention_noalloc(ctypes.byref(bad), P, 192, 3, P, 192, None) == 8   # head_dim
    kv = _kv(fg, cap=16, heads=2, d=64)
    assert L.fg_decode_attention_noalloc(ctypes.byref(kv), P, 128, 16, P, 128, None) == 4   # pos
    assert L.fg_decode_attention_noalloc(ctypes.byref(kv), P, 100, 3, P, 128, None) == 2    # ldq


def test_topk_attention_host_errors(fg):
    """fg_decode_attention_topk rejects bad arguments on the host, before any
    CUDA call (these need no GPU)."""
    L = fg.lib
    P = ctypes.c_void_p(4096)
    kv = _kv(fg, cap=16, heads=2, d=64)
    assert L.fg_decode_attention_topk(None, P, 128, 3, 2, P, 128, None, None) == 1             # null kv
    assert L.fg_decode_attention_topk(ctypes.byref(kv), P, 128, 3, 0, P, 128, None, None) == 1  # keep < 1
    assert L.fg_decode_attention_topk(ctypes.byref(kv), P, 128, 16, 2, P, 128, None, None) == 4  # pos
    assert L.fg_decode_attention_topk(ctypes.byref(kv), P, 100, 3, 2, P, 128, None, None) == 2   # ldq
    assert L.fg_decode_attention_topk(ctypes.byref(kv), P, 128, 3, 2, P, 128,
                                      ctypes.c_void_p(4098), None) == 3                          # idx alignment
    f32 = _kv(fg, cap=16, heads=2, d=64, dtype=1)
    assert L.fg_decode_attention_topk(ctypes.byref(f32), P, 128, 3, 2, P, 128, None, None) == 8
    dense = _kv(fg, cap=16, heads=2, d=64, codec=0)
    assert L.fg_decode_attention_topk(ctypes.byref(dense), P, 128, 3, 2, P, 128, None, None) == 8
    long = _kv(fg, cap=20000, heads=2, d=64)
    assert L.fg_decode_attention_topk(ctypes.byref(long), P, 128, 16384, 2, P, 128, None, None) == 8
    empty = _kv(fg, b=0, cap=16, heads=2, d=64)
    assert L.fg_decode_attention_topk(ctypes.byref(empty), None, 128, 3, 2, None, 128, None, None) == 0
    assert fg.topk_keep(528) == 53 and fg.topk_keep(530) == 53 and fg.topk_keep(1) == 1


def test_offload_host_errors(fg):
    """fg_decode_block_step_offload checks its arguments on the host first."""
    L = fg.lib
    P = ctypes.c_void_p(4096)
    lay, kv = _layer(fg, packed=True), _kv(fg)
    larr = (fg.fg_layer * 1)(lay)
    karr = (fg.fg_kv * 1)(kv)
    stage = L.fg_offload_stage_bytes(ctypes.byref(lay))
    assert stage > 0
    ws = L.fg_decode_block_workspace_bytes(ctypes.byref(lay), 2, 16)
    args = lambda st_ptr, st_bytes, pos=3: (larr, 1, P, 2, pos, karr, P, ctypes.c_void_p(4096), ws, st_ptr,
                                            st_bytes, None, None)
    assert L.fg_decode_block_step_offload(*args(None, stage)) == 5            # no stage
    assert L.fg_decode_block_step_offload(*args(P, stage - 1)) == 5           # stage too small
    assert L.fg_decode_block_step_offload(*args(ctypes.c_void_p(4096 + 16), stage)) == 3   # alignment
    assert L.fg_decode_block_step_offload(*args(P, stage, pos=16)) == 4       # pos at capacity
    nocopy = _layer(fg, packed=False)
    assert L.fg_decode_block_step_offload((fg.fg_layer * 1)(nocopy), 1, P, 2, 3, karr, P, P, ws, P, stage,
                                          None, None) == 1                     # no decode copies


def test_noalloc_scratch_bound_covers_every_cache(fg):
    """The built-in split scratch (1 MiB) holds what the split rule asks for,
    for every block size and cache capacity up to 4096 with head_dim 64 and
    128 (fg_decode_attention_workspace_bytes is pure host code)."""
    L = fg.lib
    worst = 0
    for d in (64, 128):
        for bh in range(1, 4097):
            for cap in (1, 2, 16, 100, 513, 544, 1024, 2048, 4096):
                kv = _kv(fg, b=bh, cap=cap, heads=1, d=d)
                worst = max(worst, L.fg_decode_attention_workspace_bytes(ctypes.byref(kv)))
    assert 0 < worst <= 1 << 20


def test_workspace_sizes_grow_with_tokens(fg):
    lay = _layer(fg)
    a = fg.lib.fg_prefill_workspace_bytes(ctypes.byref(lay), 2, 8)
    b = fg.lib.fg_prefill_workspace_bytes(ctypes.byref(lay), 2, 16)
    assert 0 < a < b
    assert fg.lib.fg_prefill_block_workspace_bytes(ctypes.byref(lay), 2, 8) > a


def test_wait_limit_setting(fg):
    assert fg.fg_set_wait_limit(1000) == fg.FG_WAIT_LIMIT_DEFAULT
    assert fg.fg_set_wait_limit(fg.FG_WAIT_LIMIT_DEFAULT) == 1000
