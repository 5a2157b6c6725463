"""Pins for the oracle's lightning-indexer scores and top-k selection.

Indexer and top-k: honbul.tistory.com/221 section "CSA" (a small indexer finds the blocks
most related to the current token; the Top-k Selector keeps only some compressed entries);
pogovet.com DeepSeek-V4 article, detail 4 (lightning indexer picks the top-k compressed blocks
for each query).  Score: I(t,s) = sum_h w[t,h] * ReLU(q[t,h] . k_s).
"""
import numpy as np
import pytest

import oracle


def _rng(s):
    return np.random.default_rng(s)


def test_single_head_positive_dots_is_a_gemv():
    rng = _rng(0)
    d = 32
    kh = np.abs(rng.standard_normal((100, d)))
    q = np.abs(rng.standard_normal((1, 1, d))).astype(np.float32)
    S = oracle.index_scores(q, np.ones((1, 1), np.float32), kh, [100])
    np.testing.assert_allclose(S[0], kh @ q[0, 0].astype(np.float64), rtol=1e-13)


def test_relu_pair_of_opposite_heads_gives_abs():
    # ReLU(x) + ReLU(-x) = |x| ;  a*ReLU(x) + b*ReLU(-x) splits by sign.
    rng = _rng(1)
    d = 16
    kh = rng.standard_normal((200, d))
    v = rng.standard_normal(d).astype(np.float32)
    q = np.stack([v, -v])[None]
    dots = kh @ v.astype(np.float64)
    S = oracle.index_scores(q, np.array([[1.0, 1.0]], np.float32), kh, [200])
    np.testing.assert_allclose(S[0], np.abs(dots), rtol=1e-13, atol=1e-14)
    S2 = oracle.index_scores(q, np.array([[0.25, 2.0]], np.float32), kh, [200])
    np.testing.assert_allclose(S2[0], np.where(dots > 0, 0.25 * dots, -2.0 * dots), rtol=1e-13, atol=1e-14)


def test_head_weights_are_linear_and_visibility_masks():
    rng = _rng(2)
    T, H, d, N = 3, 4, 8, 50
    q = rng.standard_normal((T, H, d)).astype(np.float32)
    w = rng.uniform(size=(T, H)).astype(np.float32)
    kh = rng.standard_normal((N, d))
    nv = [50, 17, 0]
    S = oracle.index_scores(q, w, kh, nv)
    per_head = [oracle.index_scores(q[:, h:h + 1], w[:, h:h + 1], kh, nv) for h in range(H)]
    np.testing.assert_allclose(S[0], sum(p[0] for p in per_head), rtol=1e-12)
    assert np.isneginf(S[1, 17:]).all() and np.isfinite(S[1, :17]).all()
    assert np.isneginf(S[2]).all()


def _brute_topk(row, n, k):
    order = sorted(range(n), key=lambda s: (-row[s], s))[:k]
    out = sorted(order)
    return out + [-1] * (k - len(out))


@pytest.mark.parametrize("seed", range(5))
def test_topk_matches_brute_force_sort(seed):
    rng = _rng(10 + seed)
    R, N = 6, 40
    S = rng.integers(0, 6, size=(R, N)).astype(np.float64)   # many equal scores
    S[1] = 3.0                                               # a row of all-equal scores
    S[2, :] = rng.standard_normal(N)
    nv = np.array([40, 40, 33, 5, 1, 0])
    for k in (1, 4, 7, 40, 45):
        got = oracle.topk(S, nv, k)
        for r in range(R):
            assert list(got[r]) == _brute_topk(S[r], int(nv[r]), k), (r, k)


def test_topk_k_ge_visible_returns_all_visible():
    S = np.random.default_rng(3).standard_normal((2, 30))
    got = oracle.topk(S, [30, 12], 32)
    assert list(got[0]) == list(range(30)) + [-1, -1]
    assert list(got[1]) == list(range(12)) + [-1] * 20


def test_topk_signed_zero_is_a_tie():
    S = np.array([[0.0, -0.0, 0.0, -0.0, 1.0]])
    assert list(oracle.topk(S, [5], 3)[0]) == [0, 1, 4]


# ---------------------------------------------------------- FP4 indexer queries
def _bf16(x):
    import torch
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_fp4_query_worked_example():
    from tests.golden import load
    g = load("fp4_query_worked.txt")
    d = 64
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, [int(i) for i in g["q_at"]]] = g["q"]
    qb = _bf16(q)
    qh = oracle.fp4_query(qb)
    want = np.zeros(d)
    want[[int(i) for i in g["q_at"]]] = g["q_hat"]
    np.testing.assert_array_equal(qh[0, 0], want)
    key = np.zeros((1, d))
    key[0, [int(i) for i in g["key_at"]]] = g["key"]
    S = oracle.index_scores(qh, np.array([[g["w"][0]]], np.float32), key, [1])
    assert S[0, 0] == g["expected"][0]


def test_fp4_query_of_representable_values_leaves_scores_unchanged():
    # values that already are 2^e * e2m1 with e the MX exponent of their run survive the
    # quantisation exactly, so the FP4-query scores equal the bf16-query scores
    rng = _rng(11)
    T, H, d, N = 2, 3, 64, 40
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    codes = rng.choice(mags, size=(T, H, d)) * rng.choice([-1, 1], size=(T, H, d))
    codes[..., 0] = 6.0                                  # every run of 32 has amax 6 -> e = its scale
    codes[..., 32] = -6.0
    e = rng.integers(-6, 6, size=(T, H, 2)).astype(np.float32)
    q = (codes.reshape(T, H, 2, 32) * np.exp2(e)[..., None]).reshape(T, H, d).astype(np.float32)
    kh = rng.standard_normal((N, d))
    w = rng.uniform(size=(T, H)).astype(np.float32)
    np.testing.assert_array_equal(oracle.fp4_query(q), q.astype(np.float64))
    np.testing.assert_array_equal(oracle.index_scores(oracle.fp4_query(q), w, kh, [N, 7]),
                                  oracle.index_scores(q, w, kh, [N, 7]))


def test_fp4_query_scales_each_run_of_32_on_its_own():
    # a run of large values next to a run of small ones: with one scale per head the small run
    # would round to zero; per-32 scales keep each run within half the largest E2M1 step of its
    # own scale (the step 4 -> 6 is 2 x 2^e)
    rng = _rng(12)
    d = 64
    q = np.concatenate([rng.uniform(50, 100, 32), rng.uniform(0.01, 0.02, 32)]).astype(np.float32)[None, None]
    qh = oracle.fp4_query(q)[0, 0]
    assert (qh[32:] != 0).all()
    for r in (slice(0, 32), slice(32, 64)):
        amax = np.abs(q[0, 0, r]).max()
        e = int(np.ceil(np.log2(amax / 6.0)))
        assert np.abs(qh[r] - q[0, 0, r]).max() <= 2.0 ** e
        assert set(np.unique(np.abs(qh[r]) / 2.0 ** e)) <= {0, 0.5, 1, 1.5, 2, 3, 4, 6}
