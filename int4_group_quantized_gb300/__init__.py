"""Python binding of libfg.so (argument marshalling only).

Every function here has the name of the C entry point it calls (include/fg.h)
and only turns torch tensors into pointers, sizes and the current CUDA
stream; all arithmetic runs in the library's CUDA kernels.  PyTorch provides
device memory and streams.  There is no fallback: if libfg.so is missing the
import fails.

Small holders (QuantWeight, Layer, KVCache) allocate the caller-owned buffers
the C structs point to and keep them alive.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfg.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
        "or `python -m int4_group_quantized_gb300.build` (there is no CPU fallback)")

_lib = ctypes.CDLL(LIB_PATH)

FG_OK = 0
STATUS = {0: "FG_OK", 1: "FG_ERR_ARG", 2: "FG_ERR_SHAPE", 3: "FG_ERR_ALIGN", 4: "FG_ERR_CAPACITY",
          5: "FG_ERR_WORKSPACE", 6: "FG_ERR_CUDA", 7: "FG_ERR_DEVICE_TIMEOUT", 8: "FG_ERR_UNSUPPORTED"}
FG_F16, FG_F32 = 0, 1
FG_CODEC_NONE, FG_CODEC_Q4G64 = 0, 1
FG_PACK_EXACT, FG_PACK_F16META = 0, 1
GROUP = 64


class FGError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = _lib.fg_last_error().decode()
        super().__init__(f"{where}: {STATUS.get(status, status)} ({detail})")


class fg_wmat(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("mins", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("dense", ctypes.c_void_p), ("K", ctypes.c_int64), ("N", ctypes.c_int64),
                ("packed", ctypes.c_void_p), ("packed_format", ctypes.c_int32)]


class fg_layer(ctypes.Structure):
    _fields_ = [("wq", fg_wmat), ("wk", fg_wmat), ("wv", fg_wmat), ("wo", fg_wmat), ("w1", fg_wmat),
                ("w2", fg_wmat), ("h1", ctypes.c_int64), ("h2", ctypes.c_int64),
                ("heads", ctypes.c_int32), ("codec", ctypes.c_int), ("dtype", ctypes.c_int)]


class fg_kv(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("k_mins", ctypes.c_void_p), ("k_scales", ctypes.c_void_p),
                ("v_mins", ctypes.c_void_p), ("v_scales", ctypes.c_void_p),
                ("k_dense", ctypes.c_void_p), ("v_dense", ctypes.c_void_p),
                ("b", ctypes.c_int64), ("capacity", ctypes.c_int64),
                ("heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("codec", ctypes.c_int), ("dtype", ctypes.c_int)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_INT = ctypes.c_int


def _sig(name, res, *args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_sig("fg_quantize_g64", _INT, _P, _INT, _I64, _I64, _P, _P, _P, _P)
_sig("fg_dequant_g64", _INT, _P, _P, _P, _I64, _I64, _P, _INT, _P)
_sig("fg_kv_append", _INT, ctypes.POINTER(fg_kv), _P, _P, _I64, _P)
_sig("fg_prefill_workspace_bytes", _SZ, ctypes.POINTER(fg_layer), _I64, _I64)
_sig("fg_decode_workspace_bytes", _SZ, ctypes.POINTER(fg_layer), _I64, _I64)
_sig("fg_prefill_block_workspace_bytes", _SZ, ctypes.POINTER(fg_layer), _I64, _I64)
_sig("fg_decode_block_workspace_bytes", _SZ, ctypes.POINTER(fg_layer), _I64, _I64)
_sig("fg_prefill_layer", _INT, ctypes.POINTER(fg_layer), _P, _I64, _I64, ctypes.POINTER(fg_kv), _P,
     _P, _SZ, _P)
_sig("fg_decode_step", _INT, ctypes.POINTER(fg_layer), _P, _I64, _I64, ctypes.POINTER(fg_kv), _P, _P,
     _SZ, _P)
_sig("fg_prefill_block", _INT, ctypes.POINTER(fg_layer), ctypes.c_int32, _P, _I64, _I64,
     ctypes.POINTER(fg_kv), _P, _P, _SZ, _P)
_sig("fg_decode_block_step", _INT, ctypes.POINTER(fg_layer), ctypes.c_int32, _P, _I64, _I64,
     ctypes.POINTER(fg_kv), _P, _P, _SZ, _P)
_sig("fg_sync_status", _INT, _P)
_sig("fg_status_str", ctypes.c_char_p, _INT)
_sig("fg_last_error", ctypes.c_char_p)
_sig("fg_version", ctypes.c_char_p)
_sig("fg_profile_start", _INT, ctypes.c_int32)
_sig("fg_profile_stop", _INT)
_sig("fg_profile_kernel_classes", ctypes.c_int32)
_sig("fg_profile_kernel_name", ctypes.c_char_p, ctypes.c_int32)
_sig("fg_profile_phase", _INT, ctypes.c_int32)
_sig("fg_profile_query", _INT, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64),
     ctypes.POINTER(ctypes.c_double))
_sig("fg_launch_count", ctypes.c_uint64)
_sig("fg_pack_weight_bytes", _SZ, _I64, _I64, ctypes.c_int32)
_sig("fg_pack_weight", _INT, ctypes.POINTER(fg_wmat), ctypes.c_int32, _P, _P)

lib = _lib


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return FG_F16
    if t.dtype == torch.float32:
        return FG_F32
    raise TypeError(f"activations must be float16 or float32, got {t.dtype}")


def _check(status: int, where: str) -> None:
    if status != FG_OK:
        raise FGError(status, where)


# ---- codec ---------------------------------------------------------------------

def fg_quantize_g64(x: torch.Tensor, codes: torch.Tensor, mins: torch.Tensor, scales: torch.Tensor,
                    stream=None) -> None:
    cols = x.shape[-1] if x.dim() else 0
    rows = x.numel() // cols if cols else 0
    _check(_lib.fg_quantize_g64(_ptr(x), _dt(x), rows, cols, _ptr(codes), _ptr(mins), _ptr(scales),
                                _stream(stream)), "fg_quantize_g64")


def fg_dequant_g64(codes: torch.Tensor, mins: torch.Tensor, scales: torch.Tensor, out: torch.Tensor,
                   stream=None) -> None:
    cols = out.shape[-1] if out.dim() else 0
    rows = out.numel() // cols if cols else 0
    _check(_lib.fg_dequant_g64(_ptr(codes), _ptr(mins), _ptr(scales), rows, cols, _ptr(out), _dt(out),
                               _stream(stream)), "fg_dequant_g64")


def quantize(x: torch.Tensor, stream=None):
    """Allocates (codes, mins, scales) for x [..., C] and fills them."""
    c = x.shape[-1]
    codes = torch.empty(x.shape[:-1] + (c // 2,), dtype=torch.uint8, device=x.device)
    mins = torch.empty(x.shape[:-1] + (c // GROUP,), dtype=torch.float32, device=x.device)
    scales = torch.empty_like(mins)
    fg_quantize_g64(x, codes, mins, scales, stream)
    return codes, mins, scales


def dequantize(codes, mins, scales, dtype=torch.float16, stream=None) -> torch.Tensor:
    out = torch.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=dtype, device=codes.device)
    fg_dequant_g64(codes, mins, scales, out, stream)
    return out


# ---- weights, layers, caches -------------------------------------------------------

class QuantWeight:
    """w in R^{K x N} (x . w) as stored: Q4G64 (codes/mins/scales, grouped
    along N = the output channel) or dense."""

    def __init__(self, K, N, codes=None, mins=None, scales=None, dense=None, packed=None,
                 packed_format=FG_PACK_EXACT):
        self.K, self.N = int(K), int(N)
        self.codes, self.mins, self.scales, self.dense = codes, mins, scales, dense
        self.packed = packed
        self.packed_format = int(packed_format)

    @staticmethod
    def from_dense(w: torch.Tensor, quantize_it: bool = True, stream=None, pack: bool | None = None,
                   pack_format: int = FG_PACK_EXACT) -> "QuantWeight":
        """pack (default: fp16 weights with N a multiple of 128) adds the
        decode copy the decode products read (fg_pack_weight), in pack_format."""
        K, N = w.shape
        if not quantize_it:
            return QuantWeight(K, N, dense=w.contiguous())
        codes, mins, scales = quantize(w.contiguous(), stream)
        q = QuantWeight(K, N, codes, mins, scales)
        if pack if pack is not None else (w.dtype == torch.float16 and N % 128 == 0):
            q.pack(stream, pack_format)
        return q

    def pack(self, stream=None, fmt: int = FG_PACK_EXACT) -> "QuantWeight":
        self.packed = torch.empty(fg_pack_weight_bytes(self.K, self.N, fmt), dtype=torch.uint8,
                                  device=self.codes.device)
        fg_pack_weight(self, fmt, self.packed, stream)
        self.packed_format = int(fmt)
        return self

    def struct(self) -> fg_wmat:
        return fg_wmat(_ptr(self.codes), _ptr(self.mins), _ptr(self.scales), _ptr(self.dense), self.K,
                       self.N, _ptr(self.packed), self.packed_format)

    def nbytes(self) -> int:
        """Bytes of the stored format (the packed copy is counted apart: packed_nbytes)."""
        ts = [self.codes, self.mins, self.scales, self.dense]
        return sum(t.numel() * t.element_size() for t in ts if t is not None)

    def packed_nbytes(self) -> int:
        return 0 if self.packed is None else self.packed.numel()


def fg_pack_weight_bytes(K: int, N: int, fmt: int = FG_PACK_EXACT) -> int:
    return int(_lib.fg_pack_weight_bytes(K, N, fmt))


def fg_pack_weight(w: "QuantWeight", fmt: int, packed: torch.Tensor, stream=None) -> None:
    s = w.struct()
    s.packed = None
    _check(_lib.fg_pack_weight(ctypes.byref(s), int(fmt), _ptr(packed), _stream(stream)), "fg_pack_weight")


class Layer:
    MATS = ("wq", "wk", "wv", "wo", "w1", "w2")

    def __init__(self, weights: dict, h1: int, h2: int, heads: int, quantized: bool, dtype: torch.dtype):
        self.w = weights
        self.h1, self.h2, self.heads = int(h1), int(h2), int(heads)
        self.quantized = quantized
        self.dtype = dtype
        self._s = fg_layer(*(weights[m].struct() for m in self.MATS), self.h1, self.h2, self.heads,
                           FG_CODEC_Q4G64 if quantized else FG_CODEC_NONE,
                           FG_F16 if dtype == torch.float16 else FG_F32)

    @staticmethod
    def from_dense(ws: dict, heads: int, quantized: bool = True, stream=None,
                   pack_format: int = FG_PACK_EXACT) -> "Layer":
        h1, h2 = ws["w1"].shape
        q = {m: QuantWeight.from_dense(ws[m], quantized, stream, pack_format=pack_format) for m in Layer.MATS}
        return Layer(q, h1, h2, heads, quantized, ws["wq"].dtype)

    @property
    def struct(self) -> fg_layer:
        return self._s

    def nbytes(self) -> int:
        return sum(self.w[m].nbytes() for m in self.MATS)

    def offloaded(self, stored_too: bool = True) -> "Layer":
        """The same layer with its weight arrays in pinned host memory (for
        fg_decode_block_step_offload, which streams the decode copies to the
        device layer by layer).  stored_too=False moves only the decode
        copies (the stored form stays where it is; a decode step reads only
        the copies)."""
        def host(t, move=True):
            return None if t is None else (t.cpu().pin_memory() if move else t)
        q = {m: QuantWeight(self.w[m].K, self.w[m].N, host(self.w[m].codes, stored_too),
                            host(self.w[m].mins, stored_too), host(self.w[m].scales, stored_too),
                            host(self.w[m].dense, stored_too), host(self.w[m].packed),
                            self.w[m].packed_format) for m in self.MATS}
        return Layer(q, self.h1, self.h2, self.heads, self.quantized, self.dtype)


class KVCache:
    """[b][heads][capacity][head_dim] cache, Q4G64 or dense, on `device`."""

    def __init__(self, b, heads, head_dim, capacity, quantized=True, dtype=torch.float16, device="cuda"):
        self.b, self.heads, self.head_dim, self.capacity = int(b), int(heads), int(head_dim), int(capacity)
        self.quantized, self.dtype = quantized, dtype
        shp = (self.b, self.heads, self.capacity)
        if quantized:
            self.k_codes = torch.zeros(shp + (head_dim // 2,), dtype=torch.uint8, device=device)
            self.v_codes = torch.zeros_like(self.k_codes)
            self.k_mins = torch.zeros(shp + (head_dim // GROUP,), dtype=torch.float32, device=device)
            self.k_scales = torch.zeros_like(self.k_mins)
            self.v_mins = torch.zeros_like(self.k_mins)
            self.v_scales = torch.zeros_like(self.k_mins)
            self.k_dense = self.v_dense = None
        else:
            self.k_dense = torch.zeros(shp + (head_dim,), dtype=dtype, device=device)
            self.v_dense = torch.zeros_like(self.k_dense)
            self.k_codes = self.v_codes = self.k_mins = self.k_scales = self.v_mins = self.v_scales = None
        self._s = fg_kv(_ptr(self.k_codes), _ptr(self.v_codes), _ptr(self.k_mins), _ptr(self.k_scales),
                        _ptr(self.v_mins), _ptr(self.v_scales), _ptr(self.k_dense), _ptr(self.v_dense),
                        self.b, self.capacity, self.heads, self.head_dim,
                        FG_CODEC_Q4G64 if quantized else FG_CODEC_NONE,
                        FG_F16 if dtype == torch.float16 else FG_F32)

    @property
    def struct(self) -> fg_kv:
        return self._s

    def nbytes(self) -> int:
        ts = [self.k_codes, self.v_codes, self.k_mins, self.k_scales, self.v_mins, self.v_scales,
              self.k_dense, self.v_dense]
        return sum(t.numel() * t.element_size() for t in ts if t is not None)


def _kv_array(kvs):
    arr = (fg_kv * len(kvs))(*(k.struct for k in kvs))
    return arr


def _layer_array(layers):
    return (fg_layer * len(layers))(*(l.struct for l in layers))


def fg_kv_append(kv: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, pos: int, stream=None) -> None:
    _check(_lib.fg_kv_append(ctypes.byref(kv.struct), _ptr(k_new), _ptr(v_new), int(pos), _stream(stream)),
           "fg_kv_append")


def fg_prefill_workspace_bytes(layer: Layer, b: int, s: int) -> int:
    return _lib.fg_prefill_workspace_bytes(ctypes.byref(layer.struct), int(b), int(s))


def fg_decode_workspace_bytes(layer: Layer, b: int, capacity: int) -> int:
    return _lib.fg_decode_workspace_bytes(ctypes.byref(layer.struct), int(b), int(capacity))


def fg_prefill_block_workspace_bytes(layer: Layer, b: int, s: int) -> int:
    return _lib.fg_prefill_block_workspace_bytes(ctypes.byref(layer.struct), int(b), int(s))


def fg_decode_block_workspace_bytes(layer: Layer, b: int, capacity: int) -> int:
    return _lib.fg_decode_block_workspace_bytes(ctypes.byref(layer.struct), int(b), int(capacity))


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A 256-byte aligned device buffer (torch's allocator aligns to 512)."""
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def fg_prefill_layer(layer: Layer, x: torch.Tensor, kv: KVCache, y: torch.Tensor, ws: torch.Tensor,
                     stream=None) -> None:
    b, s = x.shape[0], x.shape[1]
    _check(_lib.fg_prefill_layer(ctypes.byref(layer.struct), _ptr(x), b, s, ctypes.byref(kv.struct), _ptr(y),
                                 _ptr(ws), ws.numel(), _stream(stream)), "fg_prefill_layer")


def fg_decode_step(layer: Layer, t: torch.Tensor, pos: int, kv: KVCache, y: torch.Tensor, ws: torch.Tensor,
                   stream=None) -> None:
    _check(_lib.fg_decode_step(ctypes.byref(layer.struct), _ptr(t), t.shape[0], int(pos), ctypes.byref(kv.struct),
                               _ptr(y), _ptr(ws), ws.numel(), _stream(stream)), "fg_decode_step")


class Block:
    """Marshalled arrays of fg_layer / fg_kv for the block-level calls."""

    def __init__(self, layers: list, kvs: list):
        self.layers, self.kvs = layers, kvs
        self.larr = _layer_array(layers)
        self.karr = _kv_array(kvs)


def fg_prefill_block(block: Block, x: torch.Tensor, y: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    b, s = x.shape[0], x.shape[1]
    _check(_lib.fg_prefill_block(block.larr, len(block.layers), _ptr(x), b, s, block.karr, _ptr(y), _ptr(ws),
                                 ws.numel(), _stream(stream)), "fg_prefill_block")


def fg_decode_block_step(block: Block, t: torch.Tensor, pos: int, y: torch.Tensor, ws: torch.Tensor,
                         stream=None) -> None:
    _check(_lib.fg_decode_block_step(block.larr, len(block.layers), _ptr(t), t.shape[0], int(pos), block.karr,
                                     _ptr(y), _ptr(ws), ws.numel(), _stream(stream)), "fg_decode_block_step")


_sig("fg_graph_cache_create", _INT, ctypes.POINTER(ctypes.c_void_p))
_sig("fg_graph_cache_destroy", None, ctypes.c_void_p)
_sig("fg_graph_cache_size", _I64, ctypes.c_void_p)
_sig("fg_decode_block_step_graphed", _INT, ctypes.c_void_p, ctypes.POINTER(fg_layer), ctypes.c_int32, _P, _I64,
     _I64, ctypes.POINTER(fg_kv), _P, _P, _SZ, _P)


class GraphCache:
    """The CUDA graphs of recorded decode steps (fg_graph_cache)."""

    def __init__(self):
        h = ctypes.c_void_p()
        _check(_lib.fg_graph_cache_create(ctypes.byref(h)), "fg_graph_cache_create")
        self._h = h

    def __len__(self) -> int:
        return int(_lib.fg_graph_cache_size(self._h))

    def close(self) -> None:
        if self._h:
            _lib.fg_graph_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fg_decode_block_step_graphed(cache: GraphCache, block: Block, t: torch.Tensor, pos: int, y: torch.Tensor,
                                 ws: torch.Tensor, stream=None) -> None:
    _check(_lib.fg_decode_block_step_graphed(cache._h, block.larr, len(block.layers), _ptr(t), t.shape[0], int(pos),
                                             block.karr, _ptr(y), _ptr(ws), ws.numel(), _stream(stream)),
           "fg_decode_block_step_graphed")


_sig("fg_offload_stage_bytes", _SZ, ctypes.POINTER(fg_layer))
_sig("fg_decode_block_step_offload", _INT, ctypes.POINTER(fg_layer), ctypes.c_int32, _P, _I64, _I64,
     ctypes.POINTER(fg_kv), _P, _P, _SZ, _P, _SZ, _P, _P)


def fg_offload_stage_bytes(layer: Layer) -> int:
    return _lib.fg_offload_stage_bytes(ctypes.byref(layer.struct))


def fg_decode_block_step_offload(block: Block, t: torch.Tensor, pos: int, y: torch.Tensor, ws: torch.Tensor,
                                 stage: torch.Tensor, stream=None, copy_stream=None) -> None:
    """A decode step of a block whose layers' weights live in host memory
    (Layer.offloaded): the next layer's decode copies are copied into one half
    of `stage` on copy_stream while this layer computes from the other."""
    _check(_lib.fg_decode_block_step_offload(block.larr, len(block.layers), _ptr(t), t.shape[0], int(pos),
                                             block.karr, _ptr(y), _ptr(ws), ws.numel(), _ptr(stage), stage.numel(),
                                             _stream(stream), _stream(copy_stream if copy_stream is not None
                                                                      else stream)),
           "fg_decode_block_step_offload")


def fg_sync_status(stream=None) -> None:
    _check(_lib.fg_sync_status(_stream(stream)), "fg_sync_status")


def fg_profile_start(max_launches: int) -> None:
    _check(_lib.fg_profile_start(int(max_launches)), "fg_profile_start")


def fg_profile_phase(phase: int) -> None:
    _check(_lib.fg_profile_phase(int(phase)), "fg_profile_phase")


def fg_profile_stop(phases: int = 4) -> dict:
    """Stops launch tracing; returns {phase: {kernel class: (launches, total ms)}}."""
    st = _lib.fg_profile_stop()
    out = {}
    for p in range(phases):
        for i in range(_lib.fg_profile_kernel_classes()):
            n, ms = ctypes.c_int64(), ctypes.c_double()
            _lib.fg_profile_query(p, i, ctypes.byref(n), ctypes.byref(ms))
            if n.value:
                out.setdefault(p, {})[_lib.fg_profile_kernel_name(i).decode()] = (n.value, ms.value)
    _check(st, "fg_profile_stop")
    return out


_sig("fg_set_wait_limit", ctypes.c_uint32, ctypes.c_uint32)
FG_WAIT_LIMIT_DEFAULT = 1 << 24


def fg_set_wait_limit(polls: int) -> int:
    """Polls of every bounded device wait (process-wide); returns the previous value."""
    return int(_lib.fg_set_wait_limit(int(polls)))


def fg_launch_count() -> int:
    return int(_lib.fg_launch_count())


def fg_version() -> str:
    return _lib.fg_version().decode()


_sig("fg_linear_workspace_bytes", _SZ, _I64, _I64, _I64, _INT, _INT)
_sig("fg_linear", _INT, ctypes.POINTER(fg_wmat), _INT, _INT, _P, _I64, _P, ctypes.c_int32, _P, _P, _SZ, _P)


def fg_linear_workspace_bytes(M: int, K: int, N: int, quantized: bool, dtype: torch.dtype) -> int:
    return _lib.fg_linear_workspace_bytes(int(M), int(K), int(N), FG_CODEC_Q4G64 if quantized else FG_CODEC_NONE,
                                          FG_F16 if dtype == torch.float16 else FG_F32)


def fg_linear(w: QuantWeight, x: torch.Tensor, y: torch.Tensor, r: torch.Tensor | None = None, relu: bool = False,
              ws: torch.Tensor | None = None, stream=None) -> None:
    """y = act(x . w + r) through the library's product kernels."""
    quant = w.codes is not None
    M = x.shape[0]
    if ws is None:
        need = fg_linear_workspace_bytes(M, w.K, w.N, quant, x.dtype)
        ws = workspace(need, x.device) if need else None
    s = w.struct()
    _check(_lib.fg_linear(ctypes.byref(s), FG_CODEC_Q4G64 if quant else FG_CODEC_NONE, _dt(x), _ptr(x), M, _ptr(r),
                          1 if relu else 0, _ptr(y), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)),
           "fg_linear")


_sig("fg_decode_attention_workspace_bytes", _SZ, ctypes.POINTER(fg_kv))
_sig("fg_decode_attention", _INT, ctypes.POINTER(fg_kv), _P, _I64, _I64, _P, _I64, _P, _SZ, _P)


def fg_decode_attention_workspace_bytes(kv: KVCache) -> int:
    return _lib.fg_decode_attention_workspace_bytes(ctypes.byref(kv.struct))


def fg_decode_attention(kv: KVCache, q: torch.Tensor, pos: int, out: torch.Tensor, ws: torch.Tensor | None = None,
                        stream=None) -> None:
    """out[b][h*d:(h+1)*d] = softmax(q_h K_h^T / sqrt(d)) V_h over cache slots 0..pos."""
    if ws is None:
        need = fg_decode_attention_workspace_bytes(kv)
        ws = workspace(need, q.device) if need else None
    _check(_lib.fg_decode_attention(ctypes.byref(kv.struct), _ptr(q), q.stride(0), int(pos), _ptr(out), out.stride(0),
                                    _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)),
           "fg_decode_attention")


_sig("fg_decode_attention_noalloc", _INT, ctypes.POINTER(fg_kv), _P, _I64, _I64, _P, _I64, _P)


def fg_decode_attention_noalloc(kv: KVCache, q: torch.Tensor, pos: int, out: torch.Tensor, stream=None) -> None:
    """fg_decode_attention without a workspace, for callers that cannot
    allocate device memory: the split partials use a fixed array inside
    libfg.so (shared by all calls; overlapping calls race)."""
    _check(_lib.fg_decode_attention_noalloc(ctypes.byref(kv.struct), _ptr(q), q.stride(0), int(pos), _ptr(out),
                                            out.stride(0), _stream(stream)),
           "fg_decode_attention_noalloc")



_sig("fg_decode_attention_topk", _INT, ctypes.POINTER(fg_kv), _P, _I64, _I64, _I64, _P, _I64, _P, _P)


def fg_decode_attention_topk(kv: KVCache, q: torch.Tensor, pos: int, keep: int, out: torch.Tensor,
                             idx: torch.Tensor | None = None, stream=None) -> None:
    """Top-K sparse decode attention: per (sequence, head), only the `keep`
    highest-scoring tokens of slots 0..pos, weighted by the softmax over all
    of them.  idx (int32 [b][heads][min(keep, pos+1)]) receives the kept
    slots in ascending order when given."""
    if idx is not None and idx.dtype != torch.int32:
        raise TypeError("idx must be int32")
    _check(_lib.fg_decode_attention_topk(ctypes.byref(kv.struct), _ptr(q), q.stride(0), int(pos), int(keep),
                                         _ptr(out), out.stride(0), _ptr(idx), _stream(stream)),
           "fg_decode_attention_topk")


def topk_keep(tokens: int, percent: int = 10) -> int:
    """The page's sparse setting: the top `percent` per cent of the tokens,
    rounded up, at least one."""
    return max(1, (int(tokens) * int(percent) + 99) // 100)
