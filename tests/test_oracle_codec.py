"""CPU pins for the oracle's 4-bit group codec (FlexGen notes, section
"5. 近似方法", group-wise quantization equation, b = 4, g = 64).

The oracle is pinned to things other than itself: hand-worked groups
(tests/golden/codec_groups.txt), exact rational arithmetic (fractions), the
error bound the equation implies, and a quantize/dequantize fixed point.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import codec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "codec_groups.txt")


def _f32_bits(x):
    return int(np.array(x, dtype=np.float32).view(np.uint32))


def _records():
    recs, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition(" ")
        if key == "name":
            cur = {"name": val}
            recs.append(cur)
        else:
            cur[key] = val
    return recs


def _build(rule: str) -> np.ndarray:
    kind, *args = rule.split()
    j = np.arange(64)
    if kind == "mod16":
        return (j % 16).astype(np.float32)
    if kind == "const":
        return np.full(64, float(args[0]), np.float32)
    if kind == "alt":
        return np.where(j % 2 == 0, float(args[0]), float(args[1])).astype(np.float32)
    if kind == "list":
        x = np.zeros(64, np.float32)
        x[:len(args)] = [float(a) for a in args]
        return x
    if kind == "listfill":
        x = np.full(64, float(args[0]), np.float32)
        x[:len(args) - 1] = [float(a) for a in args[1:]]
        return x
    raise ValueError(rule)


@pytest.mark.parametrize("rec", _records(), ids=lambda r: r["name"])
def test_hand_worked_groups(rec):
    x = _build(rec["rule"])[None, :]
    for dt in (np.float32, np.float16):
        if dt == np.float16 and not np.all(np.isnan(x) | (x.astype(np.float16).astype(np.float32) == x)):
            continue
        codes, mins, scales = codec.quantize_g64(x.astype(dt))
        assert _f32_bits(mins[0, 0]) == int(rec["min"], 16), rec["name"]
        assert _f32_bits(scales[0, 0]) == int(rec["scale"], 16), rec["name"]
        assert codes[0].tobytes().hex() == rec["codes"], rec["name"]


def _exact_codes(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Per element: the exact rational u = (x - min)/(max - min) * 15 rounded
    half-to-even, and the distance of u from the nearest .5."""
    q = np.zeros(x.shape, np.int64)
    dist = np.zeros(x.shape)
    for r in range(x.shape[0]):
        for g0 in range(0, x.shape[1], 64):
            grp = [Fraction(float(v)) for v in x[r, g0:g0 + 64]]
            mn, mx = min(grp), max(grp)
            for k, v in enumerate(grp):
                u = (v - mn) / (mx - mn) * 15 if mx != mn else Fraction(0)
                fl = math.floor(u)
                frac = u - fl
                if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and fl % 2 == 1):
                    fl += 1
                q[r, g0 + k] = fl
                dist[r, g0 + k] = float(abs(u - math.floor(u) - Fraction(1, 2)))
    return q, dist


def test_random_fp16_codes_match_exact_rational():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((6, 256)) * rng.choice([0.01, 1.0, 300.0], size=(6, 1))).astype(np.float16)
    codes, mins, scales = codec.quantize_g64(x)
    q = codec.unpack_codes(codes).astype(np.int64)
    q_exact, dist = _exact_codes(x.astype(np.float64))
    near_tie = dist < 2.0 ** -20
    assert near_tie.sum() < 3
    assert np.array_equal(q[~near_tie], q_exact[~near_tie])
    # min/max are exact members of the group; scale is the correctly rounded r/15
    g = x.astype(np.float32).reshape(6, 4, 64)
    assert np.array_equal(mins, g.min(-1))
    r = (g.max(-1) - g.min(-1)).astype(np.float32)
    for a, b in zip(r.ravel(), scales.ravel()):
        assert Fraction(float(b)) == _round_f32(Fraction(float(a)) / 15)


def _round_f32(v: Fraction) -> Fraction:
    """Exact round-to-nearest-even of a rational to fp32, by comparing the
    candidates around a first guess with exact arithmetic."""
    c = np.float32(float(v))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best = None
    for cd in cands:
        d = abs(Fraction(float(cd)) - v)
        key = (d, int(np.array(cd).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, cd)
    return Fraction(float(best[1]))


def test_dequant_is_correctly_rounded_fma():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((8, 128)) * 7.3 + 1.1).astype(np.float32)
    codes, mins, scales = codec.quantize_g64(x)
    xh = codec.dequant_g64(codes, mins, scales, np.float32)
    q = codec.unpack_codes(codes)
    for r in range(x.shape[0]):
        for c in range(x.shape[1]):
            g = c // 64
            exact = Fraction(int(q[r, c])) * Fraction(float(scales[r, g])) + Fraction(float(mins[r, g]))
            assert Fraction(float(xh[r, c])) == _round_f32(exact)


def test_fma_random_cases():
    rng = np.random.default_rng(3)
    a = rng.integers(0, 16, 4000).astype(np.float32)
    b = (rng.standard_normal(4000) * 3).astype(np.float32)
    c = (rng.standard_normal(4000) * 2.0 ** rng.integers(-30, 5, 4000)).astype(np.float32)
    got = codec.fma_f32(a, b, c)
    for i in range(4000):
        exact = Fraction(float(a[i])) * Fraction(float(b[i])) + Fraction(float(c[i]))
        assert Fraction(float(got[i])) == _round_f32(exact), i


def _double_rounding_traps(count: int):
    """(q, b, c) with q*b exactly halfway between two fp32 values and c a
    nudge far below fp64 resolution that points away from the even
    neighbour: the exact sum must round away from the tie, but a plain fp64
    sum lands on the tie and a cast to fp32 then picks the even side."""
    rng = np.random.default_rng(7)
    out = []
    while len(out) < count:
        q = int(rng.choice([3, 5, 7, 9, 11, 13, 15]))
        mant = int(rng.integers(2 ** 23, 2 ** 24)) | 1
        e = int(rng.integers(-20, 20))
        b = np.float32(mant * 2.0 ** (e - 23))
        p = Fraction(q) * Fraction(float(b))
        lo = np.float32(float(p))
        if Fraction(float(lo)) > p:
            lo = np.nextafter(lo, np.float32(-np.inf))
        hi = np.nextafter(lo, np.float32(np.inf))
        if Fraction(float(lo)) + Fraction(float(hi)) != 2 * p:
            continue                                  # not a halfway case
        even_is_lo = int(np.array(lo).view(np.uint32)) % 2 == 0
        ulp64 = 2.0 ** (math.frexp(float(p))[1] - 53)
        nudge = np.float32(ulp64 / 8)
        c = nudge if even_is_lo else -nudge           # push away from the even side
        out.append((np.float32(q), b, c, hi if even_is_lo else lo))
    return out


def test_fma_double_rounding_traps():
    cases = _double_rounding_traps(200)
    a = np.array([t[0] for t in cases], np.float32)
    b = np.array([t[1] for t in cases], np.float32)
    c = np.array([t[2] for t in cases], np.float32)
    want = np.array([t[3] for t in cases], np.float32)
    naive = (a.astype(np.float64) * b + c).astype(np.float32)
    assert np.all(naive != want)                      # the trap is real
    got = codec.fma_f32(a, b, c)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    for i in range(len(cases)):
        exact = Fraction(float(a[i])) * Fraction(float(b[i])) + Fraction(float(c[i]))
        assert Fraction(float(got[i])) == _round_f32(exact)


def test_error_bound():
    """|x - x_hat| <= scale/2 + 4 ulp_f32(max(|min|, |max|)) for finite groups
    with max > min (the equation rounds to the nearest of 16 levels spaced
    (max-min)/15; the rest covers the fp32 rounding of r, scale and the fma)."""
    rng = np.random.default_rng(4)
    for std in (1e-3, 1.0, 1e3):
        x = (rng.standard_normal((16, 512)) * std).astype(np.float32)
        codes, mins, scales = codec.quantize_g64(x)
        xh = codec.dequant_g64(codes, mins, scales, np.float32).astype(np.float64)
        g = x.astype(np.float64).reshape(16, 8, 64)
        mag = np.maximum(np.abs(g.min(-1)), np.abs(g.max(-1)))
        bound = scales.astype(np.float64) / 2 + 4 * np.spacing(mag.astype(np.float32)).astype(np.float64)
        err = np.abs(g - xh.reshape(16, 8, 64)).max(-1)
        assert np.all(err <= bound)
        # the bound is tight: some element sits near half a step away
        assert np.max(err / (scales / 2)) > 0.9


def test_error_bound_fp16_output():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 256)).astype(np.float16)
    codes, mins, scales = codec.quantize_g64(x)
    xh = codec.dequant_g64(codes, mins, scales, np.float16).astype(np.float64)
    g = x.astype(np.float64).reshape(4, 4, 64)
    mag = np.maximum(np.abs(g.min(-1)), np.abs(g.max(-1)))
    bound = (scales / 2 + 4 * np.spacing(mag.astype(np.float32)))[..., None] \
        + np.spacing(np.abs(xh.reshape(4, 4, 64)).astype(np.float16)).astype(np.float64) / 2
    assert np.all(np.abs(g - xh.reshape(4, 4, 64)) <= bound)


def test_requantize_is_fixed_point():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((8, 192)).astype(np.float32)
    c1, m1, s1 = codec.quantize_g64(x)
    xh = codec.dequant_g64(c1, m1, s1, np.float32)
    c2, m2, s2 = codec.quantize_g64(xh)
    assert np.array_equal(c1, c2)
    assert np.array_equal(m1, m2)


def test_fp16_subnormal_ramp_exact():
    # x_j = j * 2^-24 (fp16 subnormals, exact in fp32): q_j = rint(15 j / 63)
    j = np.arange(64)
    x = (j * 2.0 ** -24).astype(np.float16)
    assert np.array_equal(x.astype(np.float64), j * 2.0 ** -24)
    codes, mins, scales = codec.quantize_g64(x[None])
    q = codec.unpack_codes(codes)[0]
    want = [math.floor(Fraction(15 * k, 63) + Fraction(1, 2)) for k in j]  # no ties: 10k != 21(2m+1)
    assert list(q) == want


def test_packing_layout():
    x = np.zeros((1, 64), np.float32)
    x[0, 1] = 1.0            # odd element -> high nibble of byte 0
    codes, _, _ = codec.quantize_g64(x)
    assert codes[0, 0] == 0xF0 and np.all(codes[0, 1:] == 0)
    assert np.array_equal(codec.unpack_codes(codes)[0, :2], [0, 15])


def test_all_nan_group_and_shape_errors():
    x = np.full((1, 64), np.nan, np.float32)
    codes, mins, scales = codec.quantize_g64(x)
    assert np.isnan(mins[0, 0]) and np.isnan(scales[0, 0]) and np.all(codes == 0)
    with pytest.raises(ValueError):
        codec.quantize_g64(np.zeros((2, 65), np.float32))


# ---- the opt-in fp16-metadata reading (the decode copy's FG_PACK_F16META) --------

def _all_f16_finite():
    v = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    v = np.unique(v[np.isfinite(v)].astype(np.float64))
    return v


_F16 = None


def _round_f16(x: Fraction) -> float:
    """Nearest fp16 to the exact rational x, ties to even significand, found
    by bisection in the sorted table of every finite fp16 value (no fp16
    arithmetic involved)."""
    global _F16
    if _F16 is None:
        _F16 = _all_f16_finite()
    import bisect
    i = bisect.bisect_left(_F16.tolist(), float(x))
    cands = [_F16[j] for j in (i - 1, i, i + 1) if 0 <= j < len(_F16)]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - x),
                                     int(np.float16(c).view(np.uint16)) & 1))
    return float(best)


def test_f16meta_matches_exact_rational_rounding():
    """Every element: round_f16(q * round_f16(scale) + round_f16(min)) with
    exact rationals and a table-search rounding."""
    rng = np.random.default_rng(21)
    x = np.concatenate([rng.standard_normal((2, 128)) * 0.02, rng.standard_normal((2, 128)) * 3.0,
                        rng.standard_normal((2, 128)) * 900.0]).astype(np.float16)
    codes, mins, scales = codec.quantize_g64(x)
    got = codec.dequant_g64_f16meta(codes, mins, scales)
    assert got.dtype == np.float16
    q = codec.unpack_codes(codes)
    for r in range(x.shape[0]):
        for g in range(x.shape[1] // 64):
            s16 = Fraction(_round_f16(Fraction(float(scales[r, g]))))
            m16 = Fraction(_round_f16(Fraction(float(mins[r, g]))))
            for c in range(64 * g, 64 * g + 64):
                want = _round_f16(int(q[r, c]) * s16 + m16)
                assert float(got[r, c]) == want, (r, c)


def test_f16meta_error_bound():
    """|x - w~| <= scale/2 + 15 ulp16(scale)/2 + ulp16(min)/2 + ulp16(w~)/2,
    plus the fp32 codec's own slack, for finite groups whose scale and min are
    normal fp16 numbers."""
    rng = np.random.default_rng(22)
    for std in (0.02, 1.0, 100.0):
        x = (rng.standard_normal((8, 512)) * std).astype(np.float16)
        codes, mins, scales = codec.quantize_g64(x)
        w = codec.dequant_g64_f16meta(codes, mins, scales).astype(np.float64).reshape(8, 8, 64)
        g = x.astype(np.float64).reshape(8, 8, 64)
        mag = np.maximum(np.abs(g.min(-1)), np.abs(g.max(-1)))
        ulp16 = lambda v: np.spacing(np.abs(np.asarray(v)).astype(np.float16)).astype(np.float64)
        bound = (scales / 2 + 15 * ulp16(scales) / 2 + ulp16(mins) / 2
                 + 4 * np.spacing(mag.astype(np.float32)))[..., None] + ulp16(w) / 2
        assert np.all(np.abs(g - w) <= bound)


def test_f16meta_equals_format_of_record_when_meta_is_fp16():
    """A group whose min, scale and every q*scale + min are exact fp16 values:
    both readings give the same fp16 weights."""
    j = np.arange(64)
    x = (1.0 + (j % 16) / 8.0).astype(np.float16)[None, :]   # min 1, max 2.875, scale 1/8
    codes, mins, scales = codec.quantize_g64(x)
    assert float(scales[0, 0]) == 0.125 and float(mins[0, 0]) == 1.0
    a = codec.dequant_g64_f16meta(codes, mins, scales)
    b = codec.dequant_g64(codes, mins, scales, np.float16)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    assert np.array_equal(a, x)
