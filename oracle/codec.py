"""Group-wise asymmetric 4-bit codec, written out plainly in numpy (test oracle).

Source: FlexGen notes (papercache.org, "FlexGen: High-Throughput Generative
Inference of Large Language Models with a Single GPU"), section
"5. 近似方法 (Approximate Methods)", group-wise quantization equation:
every g consecutive elements along one dimension form a group; with the
group's min and max each element x becomes the b-bit integer
round((x - min) / (max - min) * (2^b - 1)).  The same section fixes b = 4,
g = 64, weights grouped along the output channel, KV along the hidden
dimension, storage in the quantized form and conversion back to FP16
before compute.

Readings of what the page leaves open:
  * arithmetic is IEEE fp32, each operation rounded to nearest-even in the
    literal order ((x - mn) / r) * 15, no fused multiply-add;
  * "round" is round-half-to-even;
  * min and max follow the IEEE total order on the non-NaN members of the
    group (so -0 < +0); a group that is all NaN gets NaN for both;
  * codes are clamped to [0, 15] with fmax/fmin, so a NaN quotient (0/0 for
    a constant group, inf/inf) becomes code 0;
  * the scale stored beside the min is r / 15 (fp32), and the element is
    restored as the correctly rounded fp32 value of q * scale + min, then
    rounded to fp16 when the consumer computes in fp16;
  * two codes per byte, the even element in the low nibble.

This module is test infrastructure: only tests, the smoke check and the
benchmark's CPU baseline use it.  It shares nothing with the CUDA library.
"""
from __future__ import annotations

import numpy as np

GROUP = 64
LEVELS = 15  # 2^b - 1 with b = 4

_F32 = np.float32


def _group_view(x: np.ndarray) -> np.ndarray:
    if x.ndim < 1 or x.shape[-1] % GROUP != 0:
        raise ValueError("last dimension must be a multiple of 64")
    return x.reshape(x.shape[:-1] + (x.shape[-1] // GROUP, GROUP))


def group_min_max(g: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Min and max of each group (last axis) under the IEEE total order on
    non-NaN values: NaN members are skipped, -0 counts below +0, and an
    all-NaN group yields NaN."""
    nan = np.isnan(g)
    all_nan = nan.all(axis=-1)
    big = np.where(nan, np.inf, g)
    small = np.where(nan, -np.inf, g)
    mn = big.min(axis=-1)
    mx = small.max(axis=-1)
    zero = g == 0
    has_neg_zero = (zero & np.signbit(g)).any(axis=-1)
    has_pos_zero = (zero & ~np.signbit(g)).any(axis=-1)
    mn = np.where((mn == 0) & has_neg_zero, _F32(-0.0), mn)
    mn = np.where((mn == 0) & ~has_neg_zero, _F32(0.0), mn)
    mx = np.where((mx == 0) & has_pos_zero, _F32(0.0), mx)
    mx = np.where((mx == 0) & ~has_pos_zero, _F32(-0.0), mx)
    qnan = np.array(0x7FFFFFFF, dtype=np.uint32).view(np.float32)
    mn = np.where(all_nan, qnan, mn).astype(_F32)
    mx = np.where(all_nan, qnan, mx).astype(_F32)
    return mn, mx


def quantize_g64(x: np.ndarray) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Quantize along the last axis in groups of 64.

    x: float16 or float32 array [..., C] with C % 64 == 0.
    Returns (codes uint8 [..., C/2], mins float32 [..., C/64],
    scales float32 [..., C/64]).
    """
    if x.dtype not in (np.float16, np.float32):
        raise TypeError("x must be float16 or float32")
    g = _group_view(np.asarray(x).astype(_F32))  # fp16 -> fp32 is exact
    mn, mx = group_min_max(g)
    with np.errstate(all="ignore"):
        r = np.subtract(mx, mn, dtype=_F32)
        scale = np.divide(r, _F32(LEVELS), dtype=_F32)
        d = np.subtract(g, mn[..., None], dtype=_F32)
        v = np.divide(d, r[..., None], dtype=_F32)
        u = np.multiply(v, _F32(LEVELS), dtype=_F32)
        q = np.fmin(np.fmax(np.rint(u), _F32(0.0)), _F32(LEVELS))
    q = q.astype(np.uint8).reshape(x.shape)
    codes = (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)
    return codes, mn.astype(_F32), scale.astype(_F32)


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """Inverse of the nibble packing: [..., C/2] bytes -> [..., C] codes."""
    lo = codes & 0x0F
    hi = codes >> 4
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def fma_f32(a: np.ndarray, b: np.ndarray, c: np.ndarray) -> np.ndarray:
    """Correctly rounded fp32 a*b + c for fp32 inputs where a*b is exact in
    fp64 (true for a 4-bit integer times an fp32 scale).

    Method: round-to-odd (Boldo and Melquiond, "Emulation of FMA and
    correctly-rounded sums: proved algorithms using rounding to odd", IEEE
    Trans. Computers 2008): the sum is formed in fp64 rounded to odd, then
    rounded once to fp32; fp64 carries more than 24 + 2 bits, so the final
    result equals the exact sum rounded to nearest-even.
    """
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    c = np.asarray(c, dtype=np.float64)
    with np.errstate(all="ignore"):
        p = a * b                      # exact: at most 4 + 24 significant bits
        s = p + c                      # fp64, round-to-nearest-even
        bb = s - p                     # Knuth two-sum: err = exact - s
        err = (p - (s - bb)) + (c - bb)
        finite = np.isfinite(s) & np.isfinite(err)
        bits = s.view(np.int64) if s.ndim else np.array(s).view(np.int64)
        even = (bits & 1) == 0
        fix = finite & (err != 0) & even
        toward = np.where(err > 0, np.inf, -np.inf)
        s = np.where(fix, np.nextafter(s, toward), s)
    return s.astype(_F32)


def dequant_g64(codes: np.ndarray, mins: np.ndarray, scales: np.ndarray,
                out_dtype=np.float32) -> np.ndarray:
    """x_hat = fma(q, scale, min) in fp32, then rounded to out_dtype."""
    q = unpack_codes(codes).astype(_F32)
    qg = _group_view(q)
    xh = fma_f32(qg, scales[..., None].astype(_F32), mins[..., None].astype(_F32))
    xh = xh.reshape(q.shape)
    return xh.astype(out_dtype)


def dequant_g64_f16meta(codes: np.ndarray, mins: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """The opt-in fp16-metadata reading of "converted back to FP16": the
    group's scale and min are first rounded to fp16 (nearest even), then
    q * scale16 + min16 is formed exactly and rounded once to fp16.  (The
    exact value needs at most 44 significant bits -- a 4-bit integer times an
    11-bit fp16 significand, plus an fp16, all within fp16's exponent range
    -- so fp64 holds it exactly and numpy's fp64 -> fp16 cast is the single
    rounding.)  Returns float16 [..., C]."""
    q = unpack_codes(codes).astype(np.float64)
    qg = _group_view(q)
    s16 = np.asarray(scales, dtype=_F32).astype(np.float16).astype(np.float64)
    m16 = np.asarray(mins, dtype=_F32).astype(np.float16).astype(np.float64)
    with np.errstate(all="ignore"):
        exact = qg * s16[..., None] + m16[..., None]
    return exact.reshape(q.shape).astype(np.float16)


def round_trip(x: np.ndarray, out_dtype=None) -> np.ndarray:
    """dequant(quant(x)) in x's dtype (or out_dtype)."""
    c, m, s = quantize_g64(x)
    return dequant_g64(c, m, s, x.dtype if out_dtype is None else out_dtype)
