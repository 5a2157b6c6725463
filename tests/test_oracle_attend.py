"""Pins for the oracle's attention steps (CSA sparse + window, HCA dense + window, LSE merge).

CSA attends over the selected compressed entries together with a sliding window of recent raw
tokens (honbul.tistory.com/221 section "CSA"; pogovet.com article detail 4); HCA attends over
every compressed entry (honbul.tistory.com/221 section "HCA"; pogovet.com detail 4).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

import oracle


def _sdpa(q, K, V, scale):
    qt = torch.from_numpy(np.asarray(q, np.float64))[None]        # [1, H, d] -> heads as batch
    Kt = torch.from_numpy(np.asarray(K, np.float64))
    Vt = torch.from_numpy(np.asarray(V, np.float64))
    out = F.scaled_dot_product_attention(qt.transpose(0, 1), Kt[None].expand(q.shape[0], -1, -1),
                                         Vt[None].expand(q.shape[0], -1, -1), scale=scale)
    return out[:, 0].numpy()


def test_plain_attention_equals_library_sdpa():
    rng = np.random.default_rng(0)
    H, d, n = 4, 16, 50
    q = rng.standard_normal((H, d)).astype(np.float32)
    K = rng.standard_normal((n, d)).astype(np.float32)
    V = rng.standard_normal((n, d)).astype(np.float32)
    o, lse = oracle.attend(q, 0.25, K, V, np.arange(n), None, None, [])
    np.testing.assert_allclose(o, _sdpa(q, K, V, 0.25), rtol=1e-12, atol=1e-13)
    s = 0.25 * q.astype(np.float64) @ K.astype(np.float64).T
    np.testing.assert_allclose(lse, logsumexp(s, axis=1), rtol=1e-13)


def test_weights_sum_to_one_and_union_is_joint():
    rng = np.random.default_rng(1)
    H, d = 3, 8
    q = rng.standard_normal((H, d)).astype(np.float32)
    Kc = rng.standard_normal((20, d)).astype(np.float32)
    Kw = rng.standard_normal((6, d)).astype(np.float32)
    ones_c = np.ones((20, d), np.float32)
    ones_w = np.ones((6, d), np.float32)
    o, _ = oracle.attend(q, 0.3, Kc, ones_c, [1, 5, 7], Kw, ones_w, [0, 2, 3])
    np.testing.assert_allclose(o, 1.0, rtol=1e-14)
    # joint softmax over the union == plain attention over the concatenated rows
    Vc = rng.standard_normal((20, d)).astype(np.float32)
    Vw = rng.standard_normal((6, d)).astype(np.float32)
    o, lse = oracle.attend(q, 0.3, Kc, Vc, [1, 5, 7], Kw, Vw, [0, 2, 3])
    K = np.concatenate([Kc[[1, 5, 7]], Kw[[0, 2, 3]]])
    V = np.concatenate([Vc[[1, 5, 7]], Vw[[0, 2, 3]]])
    np.testing.assert_allclose(o, _sdpa(q, K, V, 0.3), rtol=1e-12, atol=1e-13)
    # permutation invariance of the compressed row list
    o2, lse2 = oracle.attend(q, 0.3, Kc, Vc, [7, 1, 5], Kw, Vw, [3, 0, 2])
    np.testing.assert_allclose(o2, o, rtol=1e-13, atol=1e-14)


def test_split_merge_equals_single_pass():
    rng = np.random.default_rng(2)
    H, d, n = 5, 12, 97
    q = rng.standard_normal((H, d)).astype(np.float32)
    K = rng.standard_normal((n, d)).astype(np.float32) * 3
    V = rng.standard_normal((n, d)).astype(np.float32)
    o, lse = oracle.attend(q, 0.5, K, V, np.arange(n), None, None, [])
    cuts = [0, 10, 11, 50, 97]
    parts = [oracle.attend(q, 0.5, K, V, np.arange(a, b), None, None, []) for a, b in zip(cuts, cuts[1:])]
    parts.append(oracle.attend(q, 0.5, K, V, [], None, None, []))     # an empty split
    om, lm = oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(om, o, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lm, lse, rtol=1e-14)


def _toy_sequence(rng, L, d, m):
    K = rng.standard_normal((L, d)).astype(np.float32)
    V = rng.standard_normal((L, d)).astype(np.float32)
    gate = rng.standard_normal(L).astype(np.float32)
    bias = (0.5 * rng.standard_normal(m)).astype(np.float32)
    return K, V, gate, bias


def test_csa_with_k_ge_visible_equals_dense_hca_form():
    # k >= number of visible compressed entries => CSA == dense attention over all visible
    # compressed entries plus the window (the HCA form with the same m).
    rng = np.random.default_rng(3)
    L, d, H, m, W, HI, dI = 203, 16, 4, 4, 9, 2, 8
    K, V, gate, bias = _toy_sequence(rng, L, d, m)
    ck, cv = oracle.compress(K, V, gate, bias, m, oracle.F32)
    n = ck.shape[0]
    kin = rng.standard_normal((n, dI)).astype(np.float32)
    q = rng.standard_normal((3, H, d)).astype(np.float32)
    qi = rng.standard_normal((3, HI, dI)).astype(np.float32)
    w = rng.uniform(size=(3, HI)).astype(np.float32)
    pos = np.array([L - 1, 120, 3])
    csa = oracle.csa_queries(q, qi, w, pos, ck, cv, kin, None, oracle.KEY_F32, K, V, 0, m, n + 5, W, 0.25)
    hca = oracle.hca_queries(q, pos, ck, cv, K, V, 0, m, W, 0.25)
    np.testing.assert_allclose(csa["o"], hca["o"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(csa["lse"], hca["lse"], rtol=1e-13)
    assert list(csa["idx"][1][:30]) == list(range(30)) and csa["idx"][1][30] == -1


def test_hca_with_m1_no_window_is_full_causal_attention():
    rng = np.random.default_rng(4)
    L, d, H = 64, 8, 3
    K, V, gate, _ = _toy_sequence(rng, L, d, 1)
    ck, cv = oracle.compress(K, V, np.zeros(L, np.float32), np.zeros(1, np.float32), 1, oracle.F32)
    q = rng.standard_normal((4, H, d)).astype(np.float32)
    pos = np.array([63, 0, 31, 40])
    res = oracle.hca_queries(q, pos, ck, cv, K, V, 0, 1, 0, 0.35)
    for t, p in enumerate(pos):
        np.testing.assert_allclose(res["o"][t], _sdpa(q[t], K[:p + 1], V[:p + 1], 0.35), rtol=1e-12, atol=1e-13)


def test_csa_with_k0_is_sliding_window_attention():
    rng = np.random.default_rng(5)
    L, d, H, m, W = 80, 8, 2, 4, 16
    K, V, gate, bias = _toy_sequence(rng, L, d, m)
    ck, cv = oracle.compress(K, V, gate, bias, m, oracle.F32)
    kin = rng.standard_normal((ck.shape[0], 8)).astype(np.float32)
    q = rng.standard_normal((2, H, d)).astype(np.float32)
    qi = rng.standard_normal((2, 1, 8)).astype(np.float32)
    pos = np.array([79, 5])
    res = oracle.csa_queries(q, qi, np.ones((2, 1), np.float32), pos, ck, cv, kin, None,
                             oracle.KEY_F32, K, V, 0, m, 0, W, 0.4)
    for t, p in enumerate(pos):
        lo = max(0, p - W + 1)
        np.testing.assert_allclose(res["o"][t], _sdpa(q[t], K[lo:p + 1], V[lo:p + 1], 0.4), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("strict", [False, True])
def test_visibility_rule(strict):
    # causally complete: entry j visible at p iff (j+1)*m <= p+1 ; strict: (j+1)*m <= p
    m = 4
    for p in range(0, 20):
        n = oracle.n_visible(p, m, strict=strict)
        want = sum(1 for j in range(10) if (j + 1) * m <= (p if strict else p + 1))
        assert n == want
