"""GPU parity of the codec kernels (fg_quantize_g64, fg_dequant_g64,
fg_kv_append) against the oracle: codes, mins and scales bit-exact, dequant
output bit-exact (FlexGen notes, "5. 近似方法")."""
import numpy as np
import pytest
import torch

import synth
from oracle import codec as ocodec
from tests.test_oracle_codec import _build, _records

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fg():
    import int4_group_quantized_gb300 as fg
    return fg


def _bits(a):
    return np.asarray(a).view(np.uint32)


def _check_quant(fg, x: torch.Tensor):
    codes, mins, scales = fg.quantize(x)
    torch.cuda.synchronize()
    oc, om, os_ = ocodec.quantize_g64(x.cpu().numpy())
    assert np.array_equal(codes.cpu().numpy(), oc)
    gm, gs = mins.cpu().numpy(), scales.cpu().numpy()
    nan_m = np.isnan(om)
    assert np.array_equal(np.isnan(gm), nan_m) and np.array_equal(_bits(gm)[~nan_m], _bits(om)[~nan_m])
    nan_s = np.isnan(os_)
    assert np.array_equal(np.isnan(gs), nan_s) and np.array_equal(_bits(gs)[~nan_s], _bits(os_)[~nan_s])
    return codes, mins, scales, (oc, om, os_)


@pytest.mark.parametrize("dtype", [torch.float16, torch.float32])
@pytest.mark.parametrize("shape", [(1, 64), (3, 128), (7, 192), (129, 320), (1000, 64 * 9)])
def test_quantize_dequant_random(fg, dtype, shape):
    x = synth.normal(shape, 11 + shape[0], 1.0, dtype, "cuda")
    codes, mins, scales, (oc, om, os_) = _check_quant(fg, x)
    for odt, ont in ((torch.float32, np.float32), (torch.float16, np.float16)):
        out = fg.dequantize(codes, mins, scales, odt)
        ref = ocodec.dequant_g64(oc, om, os_, ont)
        assert np.array_equal(out.cpu().numpy().view(np.uint8), ref.view(np.uint8))


@pytest.mark.parametrize("rec", _records(), ids=lambda r: r["name"])
def test_hand_worked_groups(fg, rec):
    x = torch.from_numpy(_build(rec["rule"])[None, :].copy()).cuda()
    codes, mins, scales = fg.quantize(x)
    assert int(np.array(mins.cpu().numpy()[0, 0]).view(np.uint32)) == int(rec["min"], 16)
    assert int(np.array(scales.cpu().numpy()[0, 0]).view(np.uint32)) == int(rec["scale"], 16)
    assert codes.cpu().numpy()[0].tobytes().hex() == rec["codes"]


def test_special_values(fg):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((16, 128)).astype(np.float32)
    x[0, :64] = np.nan                        # all-NaN group
    x[1, 3] = np.nan                          # one NaN member
    x[2, 7] = np.inf
    x[3, 9] = -np.inf
    x[4, :] = 0.0
    x[4, 1::2] = -0.0                         # signed zeros
    x[5, :64] = 2.5                           # constant group
    x[6, :] = x[6, :] * 1e30                  # huge range, fp32 only
    x[7, :] = x[7, :] * 1e-40                 # fp32 subnormals
    x[8, :64] = np.where(np.arange(64) % 2 == 0, 3.0, -7.0)
    x[9, 0], x[9, 1] = np.finfo(np.float32).max, -np.finfo(np.float32).max  # r overflows to inf
    _check_quant(fg, torch.from_numpy(x).cuda())
    h = rng.standard_normal((8, 128)).astype(np.float16)
    h[0, :] = (np.arange(128) % 64 * 2.0 ** -24).astype(np.float16)     # fp16 subnormals
    h[1, :] = np.float16(65504.0) * np.sign(rng.standard_normal(128)).astype(np.float16)
    h[2, :64] = np.float16(-0.0)
    h[3, 5] = np.float16(np.nan)
    _check_quant(fg, torch.from_numpy(h).cuda())


@pytest.mark.parametrize("name", ["opt-125m", "opt-6.7b", "opt-30b", "opt-175b"])
def test_weight_shapes(fg, name):
    """Every weight shape of the OPT workloads; the largest matrices are
    checked on a sample of rows (rows quantize independently)."""
    w = synth.WORKLOADS[name]
    for i, m in enumerate(synth.MATS):
        K, N = synth.weight_shape(w, m)
        x = synth.normal((K, N), synth.weight_seed(w.cfg_id, 0, i), synth.WEIGHT_STD, torch.float16, "cuda")
        codes, mins, scales = fg.quantize(x)
        rows = np.unique(np.concatenate([np.arange(min(K, 8)), np.random.default_rng(i).integers(0, K, 24),
                                         [K - 1]]))
        xs = x[rows].cpu().numpy()
        oc, om, os_ = ocodec.quantize_g64(xs)
        assert np.array_equal(codes[rows].cpu().numpy(), oc), m
        assert np.array_equal(_bits(mins[rows].cpu().numpy()), _bits(om)), m
        assert np.array_equal(_bits(scales[rows].cpu().numpy()), _bits(os_)), m
        out = fg.dequantize(codes[rows].contiguous(), mins[rows].contiguous(), scales[rows].contiguous())
        ref = ocodec.dequant_g64(oc, om, os_, np.float16)
        assert np.array_equal(out.cpu().numpy().view(np.uint16), ref.view(np.uint16)), m
        del x, codes, mins, scales


def test_empty_and_errors(fg):
    x = torch.empty((0, 64), dtype=torch.float16, device="cuda")
    c, m, s = fg.quantize(x)
    assert c.shape == (0, 32)
    with pytest.raises(fg.FGError) as e:
        fg.quantize(torch.zeros((2, 96), dtype=torch.float16, device="cuda"))
    assert e.value.status == 2


@pytest.mark.parametrize("dtype,d", [(torch.float16, 128), (torch.float32, 64), (torch.float16, 64)])
def test_kv_append_bit_exact(fg, dtype, d):
    b, heads, cap = 3, 4, 10
    kv = fg.KVCache(b, heads, d, cap, True, dtype)
    rng = np.random.default_rng(d)
    ks, vs = {}, {}
    for pos in (0, 4, cap - 1):
        k = synth.normal((b, heads * d), 100 + pos, 1.0, dtype, "cuda")
        v = synth.normal((b, heads * d), 200 + pos, 1.0, dtype, "cuda")
        fg.fg_kv_append(kv, k, v, pos)
        ks[pos], vs[pos] = k.cpu().numpy(), v.cpu().numpy()
    torch.cuda.synchronize()
    for pos in ks:
        for name, rows in (("k", ks[pos]), ("v", vs[pos])):
            r = rows.reshape(b, heads, d)
            oc, om, os_ = ocodec.quantize_g64(r)
            assert np.array_equal(getattr(kv, name + "_codes")[:, :, pos].cpu().numpy(), oc)
            assert np.array_equal(_bits(getattr(kv, name + "_mins")[:, :, pos].cpu().numpy()), _bits(om))
            assert np.array_equal(_bits(getattr(kv, name + "_scales")[:, :, pos].cpu().numpy()), _bits(os_))
    # untouched slots stay zero
    assert int(kv.k_codes[:, :, 1].abs().sum()) == 0
    with pytest.raises(fg.FGError) as e:
        fg.fg_kv_append(kv, k, v, cap)
    assert e.value.status == 4
