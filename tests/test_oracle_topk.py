"""Pins for the oracle's top-K sparse decode attention (FlexGen notes,
"5. 近似方法", sparse attention: after the attention matrix, keep each query's
Top-K tokens and read only those rows of V).

Each test ties oracle.layer.attention_topk to something other than itself:
a hand-worked example in closed form (scale, tie rule, no renormalisation),
torch's fp64 scaled_dot_product_attention when every token is kept, a
brute-force rank count written with explicit loops, and properties any
top-K selection of a probability vector has."""
import math

import numpy as np
import pytest
import torch

from oracle import layer as olayer


def test_keep_count_is_ten_percent_rounded_up():
    # integers worked by hand: ceil(T / 10), at least one token
    for T, want in [(1, 1), (9, 1), (10, 1), (11, 2), (100, 10), (513, 52), (528, 53), (530, 53),
                    (531, 54), (544, 55)]:
        assert olayer.topk_keep(T) == want, T
    assert olayer.topk_keep(7, 100) == 7 and olayer.topk_keep(7, 50) == 4


def test_hand_worked_example_with_a_tie():
    # d = 2, one query q = (1, 0); keys k0 = (1, 0), k1 = (2, 0), k2 = (0, 0),
    # k3 = (2, 0): scores 1/sqrt2, sqrt2, 0, sqrt2.  Tokens 1 and 3 tie; the
    # lower index ranks first.
    q = np.array([[[1.0, 0.0]]])
    k = np.array([[[[1.0, 0.0], [2.0, 0.0], [0.0, 0.0], [2.0, 0.0]]]])
    v = np.array([[[[10.0, -1.0], [1.0, 2.0], [-3.0, 5.0], [7.0, 7.0]]]])
    r2 = math.sqrt(2.0)
    z = math.exp(1.0 / r2) + 2.0 * math.exp(r2) + 1.0
    p = [math.exp(1.0 / r2) / z, math.exp(r2) / z, 1.0 / z, math.exp(r2) / z]
    # keep 1: token 1 alone, with its weight from the softmax over all four
    out, idx = olayer.attention_topk(q, k, v, 1)
    assert idx.tolist() == [[[1]]]
    np.testing.assert_allclose(out[0, 0], [p[1] * 1.0, p[1] * 2.0], rtol=1e-14)
    # keep 2: tokens 1 and 3
    out, idx = olayer.attention_topk(q, k, v, 2)
    assert idx.tolist() == [[[1, 3]]]
    np.testing.assert_allclose(out[0, 0], [p[1] * 1 + p[3] * 7, p[1] * 2 + p[3] * 7], rtol=1e-14)
    # keep 3: then token 0 (score 1/sqrt2 > 0)
    out, idx = olayer.attention_topk(q, k, v, 3)
    assert idx.tolist() == [[[0, 1, 3]]]
    np.testing.assert_allclose(out[0, 0], [p[0] * 10 + p[1] * 1 + p[3] * 7, -p[0] + p[1] * 2 + p[3] * 7],
                               rtol=1e-14)


@pytest.mark.parametrize("T", [1, 5, 33])
def test_keeping_every_token_is_dense_attention(T):
    rng = np.random.default_rng(T)
    b, H, d = 2, 3, 16
    q = rng.normal(size=(b, H, d))
    k = rng.normal(size=(b, H, T, d))
    v = rng.normal(size=(b, H, T, d))
    want = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, :, None, :], torch.from_numpy(k), torch.from_numpy(v))[:, :, 0, :].numpy()
    for keep in (T, T + 7):
        out, idx = olayer.attention_topk(q, k, v, keep)
        np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-13)
        assert (idx == np.arange(T)).all()


def _brute(q, k, v, keep):
    """Explicit loops: a token is kept iff fewer than `keep` tokens outrank
    it (a higher score, or an equal score at a lower index)."""
    b, H, T, d = k.shape
    out = np.zeros((b, H, d))
    sets = []
    for bi in range(b):
        for h in range(H):
            s = [sum(q[bi, h, j] * k[bi, h, t, j] for j in range(d)) / math.sqrt(d) for t in range(T)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = sum(e)
            kept = []
            for t in range(T):
                rank = sum(1 for u in range(T) if s[u] > s[t] or (s[u] == s[t] and u < t))
                if rank < keep:
                    kept.append(t)
                    for j in range(d):
                        out[bi, h, j] += e[t] / z * v[bi, h, t, j]
            sets.append(kept)
    return out, sets


@pytest.mark.parametrize("T,keep", [(7, 1), (12, 3), (20, 2), (20, 19)])
def test_matches_brute_force_rank_count(T, keep):
    rng = np.random.default_rng(100 + T + keep)
    b, H, d = 2, 2, 4
    q = rng.normal(size=(b, H, d))
    k = rng.normal(size=(b, H, T, d))
    k[0, 0, 3] = k[0, 0, 5]           # an exact tie
    v = rng.normal(size=(b, H, T, d))
    out, idx = olayer.attention_topk(q, k, v, keep)
    want, sets = _brute(q, k, v, keep)
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-14)
    assert [list(r) for r in idx.reshape(b * H, -1)] == sets


def test_selection_properties():
    rng = np.random.default_rng(7)
    b, H, T, d = 3, 4, 50, 8
    q = rng.normal(size=(b, H, d)) * 2
    k = rng.normal(size=(b, H, T, d))
    ones = np.ones((b, H, T, 1))                      # v = 1: out is the kept mass
    prev = np.zeros((b, H))
    for keep in (1, 5, 17, 50):
        mass, idx = olayer.attention_topk(q, k, ones, keep)
        mass = mass[..., 0]
        # the top-K of a distribution holds at least the average share keep/T, at most all
        assert (mass >= keep / T - 1e-12).all() and (mass <= 1 + 1e-12).all()
        assert (mass >= prev - 1e-12).all()          # more tokens, more mass
        prev = mass
        # every kept score is >= every dropped score
        s = np.einsum("bhd,bhtd->bht", q, k)
        for bi in range(b):
            for h in range(H):
                kept = np.zeros(T, bool)
                kept[idx[bi, h]] = True
                if keep < T:
                    assert s[bi, h, kept].min() >= s[bi, h, ~kept].max()
    # keep 1: the largest weight times its value row
    out1, idx1 = olayer.attention_topk(q, k, k, 1)
    s = np.einsum("bhd,bhtd->bht", q, k) / np.sqrt(d)
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    am = s.argmax(-1)
    assert (idx1[..., 0] == am).all()
    want = np.take_along_axis(p, am[..., None], -1) * np.take_along_axis(k, am[..., None, None], 2)[:, :, 0]
    np.testing.assert_allclose(out1, want, rtol=1e-13)
