"""GPU parity of fg_decode_attention_topk (FlexGen notes, "5. 近似方法", sparse
attention: keep each query's Top-K tokens, read only their V rows) against
oracle.layer.attention_topk over the same cache contents.

The cache is filled through fg_kv_append (bit-exact against the oracle's
codec), so both sides hold the same 4-bit codes and restore the same fp16
K/V values.  The kernel takes its integer decision (which tokens are kept)
on fp32 scores from exact fp16 products; the oracle on fp64 scores.  So:
  * where a row's keep-th and (keep+1)-th oracle scores are further apart
    than twice the fp32 accumulation bound, the kept set is unique and must
    equal the oracle's exactly;
  * elsewhere (near-ties at the boundary) the kernel's set must be a valid
    top-K: every token that beats the boundary by more than the bound is
    kept, every token below it by more than the bound is dropped, and the
    count is keep.  Such rows are counted and must be rare;
  * the output is compared with the sum over the kernel's kept set of the
    oracle's softmax weights times the oracle's values (on rows with the
    oracle's set, exactly the oracle's output): max|d|/max|ref| <= 5e-3.
A case with integer K values and heavy exact ties checks the tie rule (lower
slot first) with no tolerance at all."""
import numpy as np
import pytest
import torch

import synth
from oracle import layer as olayer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fg():
    import int4_group_quantized_gb300 as fg
    return fg


def _fill(fg, b, H, d, length, cap, k, v, rows=None):
    """The GPU cache of all b sequences; the oracle's of the sequences `rows`
    (all by default; sequences are independent)."""
    kv = fg.KVCache(b, H, d, cap, True, torch.float16, "cuda")
    for p in range(length):
        fg.fg_kv_append(kv, k[p].contiguous(), v[p].contiguous(), p)
    rows = list(range(b)) if rows is None else rows
    oc = olayer.KVCache(len(rows), H, d, cap, True, "f16")
    oc.store(k[:, rows].cpu().numpy().astype(np.float64).transpose(1, 0, 2),
             v[:, rows].cpu().numpy().astype(np.float64).transpose(1, 0, 2), 0)
    return kv, oc


def _run(fg, kv, q, pos, keep):
    b, h1 = q.shape
    H = kv.struct.heads
    out = torch.full_like(q, float("nan"))
    kk = min(keep, pos + 1)
    idx = torch.full((b, H, kk), -1, dtype=torch.int32, device="cuda")
    fg.fg_decode_attention_topk(kv, q, pos, keep, out, idx)
    fg.fg_sync_status()
    return out.cpu().numpy().astype(np.float64), idx.cpu().numpy()


def _check(q, oc, length, keep, out, idx, min_unique=0.95):
    b, H, d = oc.b, oc.heads, oc.head_dim
    qo = q.cpu().numpy().astype(np.float64).reshape(b, H, d)
    out = out[:b]
    idx = idx[:b]
    k = oc.k_val[:, :, :length]
    v = oc.v_val[:, :, :length]
    want, widx = olayer.attention_topk(qo, k, v, keep)
    # the oracle's own softmax weights, for the kernel's kept sets
    s = np.einsum("bhd,bhtd->bht", qo, k) / np.sqrt(d)
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    # fp32 accumulation bound of a score (exact fp16 products; generous)
    bound = 2.0 ** -18 * np.einsum("bhd,bhtd->bht", np.abs(qo), np.abs(k)).max(-1) / np.sqrt(d) + 1e-30
    kk = min(keep, length)
    ref = np.zeros((b, H, d))
    unique = ambiguous = 0
    for bi in range(b):
        for h in range(H):
            sel = idx[bi, h]
            assert len(set(sel.tolist())) == kk and (np.diff(sel) > 0).all(), (bi, h, sel)
            assert sel.min() >= 0 and sel.max() < length
            E = 2.0 * bound[bi, h]
            if kk < length:
                srt = np.sort(s[bi, h])[::-1]
                sk, sk1 = srt[kk - 1], srt[kk]
                kept = np.zeros(length, bool)
                kept[sel] = True
                assert kept[s[bi, h] > sk1 + E].all(), (bi, h)
                assert not kept[s[bi, h] < sk - E].any(), (bi, h)
                if sk - sk1 > E:
                    unique += 1
                    assert (sel == widx[bi, h]).all(), (bi, h)
                else:
                    ambiguous += 1
            else:
                unique += 1
                assert (sel == np.arange(length)).all()
            ref[bi, h] = p[bi, h, sel] @ v[bi, h, sel]
            if (sel == widx[bi, h]).all():
                np.testing.assert_array_equal(ref[bi, h], want[bi, h])
    assert unique >= min_unique * (unique + ambiguous), (unique, ambiguous)
    got = out.reshape(b, H, d)
    err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert err <= 5e-3, f"rel err {err}"
    return unique, ambiguous


CASES = [
    # (b, heads, head_dim, filled slots, capacity, keep)
    (2, 4, 128, 300, 320, 30),      # the page's 10%
    (3, 2, 64, 77, 80, 8),          # ragged last block, head_dim 64
    (1, 1, 128, 1, 8, 1),           # a single cached token
    (2, 3, 128, 200, 200, 200),     # keep = every token: dense attention
    (2, 2, 64, 100, 100, 500),      # keep above the token count
    (2, 2, 128, 50, 64, 1),         # keep one: the argmax
    (2, 2, 128, 2000, 2048, 200),   # several score blocks per warp
    (64, 32, 128, 528, 544, 53),    # OPT-6.7B shape at the page's 10% (one decode step)
]
# the oracle's cache for these sequences only at the full block (its codec
# over all 64 takes minutes); the GPU attends over all of them
SAMPLE = {64: [0, 17, 40, 63]}


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b%d_H%d_d%d_len%d_keep%d" % (c[0], c[1], c[2], c[3], c[5]))
def test_topk_attention_matches_oracle(fg, case):
    b, H, d, length, cap, keep = case
    h1 = H * d
    k = synth.normal((length, b, h1), 41 + length, 1.3, torch.float16, "cuda")
    v = synth.normal((length, b, h1), 42 + length, 1.3, torch.float16, "cuda")
    rows = SAMPLE.get(b)
    kv, oc = _fill(fg, b, H, d, length, cap, k, v, rows)
    q = synth.normal((b, h1), 43, 1.3, torch.float16, "cuda")
    out, idx = _run(fg, kv, q, length - 1, keep)
    if rows is not None:
        q, out, idx = q[rows], out[rows], idx[rows]
    _check(q, oc, length, keep, out, idx)


def test_topk_attention_keep_all_equals_dense(fg):
    b, H, d, length = 2, 4, 128, 257
    h1 = H * d
    k = synth.normal((length, b, h1), 51, 1.3, torch.float16, "cuda")
    v = synth.normal((length, b, h1), 52, 1.3, torch.float16, "cuda")
    kv, oc = _fill(fg, b, H, d, length, length, k, v)
    q = synth.normal((b, h1), 53, 1.3, torch.float16, "cuda")
    out, _ = _run(fg, kv, q, length - 1, length)
    want = olayer.attention(q.cpu().numpy().astype(np.float64).reshape(b, 1, H, d), oc.k_val, oc.v_val,
                            np.array([length - 1])).reshape(b, h1)
    assert np.max(np.abs(out - want)) / np.max(np.abs(want)) <= 5e-3


@pytest.mark.parametrize("d", [64, 128])
def test_topk_ties_go_to_the_lower_slot(fg, d):
    """Integer K values (each 64-group spans 0..15, so scale 1 and min 0 and
    the codes are the values) and integer q: every score is an exact integer
    on both sides, and tokens drawn from a pool of six K rows tie exactly.
    The kept sets must equal the oracle's, ties resolved to the lower slot."""
    b, H, length, keep = 2, 2, 150, 40
    h1 = H * d
    rng = np.random.default_rng(d)
    pool = rng.integers(0, 16, size=(6, h1)).astype(np.float64)
    pool[:, 0::64] = 0.0
    pool[:, 1::64] = 15.0
    pick = rng.integers(0, 6, size=(length, b))
    kn = torch.from_numpy(pool[pick]).to(torch.float16).cuda()
    v = synth.normal((length, b, h1), 61, 1.3, torch.float16, "cuda")
    kv, oc = _fill(fg, b, H, d, length, length, kn, v)
    assert (oc.k_scales == 1.0).all() and (oc.k_mins == 0.0).all()
    q = torch.from_numpy(rng.integers(-2, 3, size=(b, h1)).astype(np.float64)).to(torch.float16).cuda()
    out, idx = _run(fg, kv, q, length - 1, keep)
    qo = q.cpu().numpy().astype(np.float64).reshape(b, H, d)
    want, widx = olayer.attention_topk(qo, oc.k_val[:, :, :length], oc.v_val[:, :, :length], keep)
    np.testing.assert_array_equal(idx, widx)
    s = np.einsum("bhd,bhtd->bht", qo, oc.k_val[:, :, :length])
    srt = np.sort(s, -1)[..., ::-1]
    assert (srt[..., keep - 1] == srt[..., keep]).any(), "no tie at the boundary"
    err = np.max(np.abs(out.reshape(b, H, d) - want)) / np.max(np.abs(want))
    assert err <= 5e-3, f"rel err {err}"


def test_topk_attention_is_repeatable(fg):
    b, H, d, length, keep = 4, 8, 128, 400, 40
    h1 = H * d
    k = synth.normal((length, b, h1), 71, 1.3, torch.float16, "cuda")
    v = synth.normal((length, b, h1), 72, 1.3, torch.float16, "cuda")
    kv, _ = _fill(fg, b, H, d, length, length, k, v)
    q = synth.normal((b, h1), 73, 1.3, torch.float16, "cuda")
    o1, i1 = _run(fg, kv, q, length - 1, keep)
    o2, i2 = _run(fg, kv, q, length - 1, keep)
    assert np.array_equal(o1, o2) and np.array_equal(i1, i2)


def test_topk_attention_without_idx_and_errors(fg):
    b, H, d, length = 2, 2, 64, 20
    kv = fg.KVCache(b, H, d, 32, True, torch.float16, "cuda")
    q = torch.zeros((b, H * d), dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    fg.fg_decode_attention_topk(kv, q, length - 1, 3, out)   # idx omitted
    fg.fg_sync_status()
    assert torch.isfinite(out).all()
    with pytest.raises(fg.FGError) as e:
        fg.fg_decode_attention_topk(kv, q, 32, 3, out)
    assert e.value.status == 4
    with pytest.raises(fg.FGError) as e:
        fg.fg_decode_attention_topk(kv, q, 5, 0, out)
    assert e.value.status == 1
