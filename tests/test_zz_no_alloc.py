"""hca_attend_noalloc: the HCA attention entry point for callers that cannot allocate device
memory (its split partials live in a fixed array inside the library instead of a caller
workspace).  Checked through the C-ABI against hca_attend on the same inputs, on two calls in
a row (the second call reuses the scratch the first one left behind).

This file is named to be collected last, so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests.gpu_cases import assert_close, npy

pytestmark = pytest.mark.gpu


def _case(seed, B=3, H=64, d=128, dtype=torch.bfloat16, Ncap=70, W=128, m=128):
    g = torch.Generator().manual_seed(seed)
    mk = lambda *s, std=1.0: (torch.randn(*s, generator=g) * std).to(dtype).cuda()  # noqa: E731
    ck, cv = mk(B, Ncap, d), mk(B, Ncap, d)
    rk, rv = mk(B, W, d), mk(B, W, d)
    q = mk(B, 1, H, d, std=d ** -0.5)
    pos = torch.tensor([m * (Ncap - 1) + 7, 300, m * 20 + 127][:B], dtype=torch.int64, device="cuda")
    return q, ck, cv, rk, rv, pos


def _oracle_rows(q, ck, cv, rk, rv, pos, m, W, d):
    """The oracle's HCA result per query row; the window comes from the ring (token t in slot
    t % W)."""
    o, lse = [], []
    for b in range(q.shape[0]):
        p = int(pos[b])
        lo = max(0, p - W + 1)
        slots = np.arange(lo, p + 1) % W
        raw_k, raw_v = npy(rk[b])[slots], npy(rv[b])[slots]
        res = oracle.hca_queries(npy(q[b]), [p], npy(ck[b]), npy(cv[b]), raw_k, raw_v, lo, m, W, d ** -0.5)
        o.append(res["o"][0])
        lse.append(res["lse"][0])
    return np.stack(o)[:, None], np.stack(lse)[:, None]


@pytest.mark.parametrize("dtype,H,d", [(torch.bfloat16, 64, 128), (torch.float32, 8, 64)])
def test_noalloc_matches_hca_attend_twice(dtype, H, d):
    import long_context_sparse_28_b300 as L
    m, W = 128, 128
    for call, seed in enumerate((1, 2)):                      # two calls in a row
        q, ck, cv, rk, rv, pos = _case(seed, H=H, d=d, dtype=dtype)
        ref = torch.empty_like(q)
        ref_lse = torch.empty(q.shape[:3], device="cuda")
        L.hca_attend(q, d ** -0.5, ck, cv, m, rk, rv, W, pos, ref, ref_lse)
        out = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:3], float("nan"), device="cuda")
        L.hca_attend_noalloc(q, d ** -0.5, ck, cv, m, rk, rv, W, pos, out, lse)
        torch.cuda.synchronize()
        assert L.device_status() == 0
        kind = "f32" if dtype == torch.float32 else "bf16"
        assert_close(out, oracle.to_f64(npy(ref)), kind, f"call {call}")
        np.testing.assert_allclose(npy(lse), npy(ref_lse), rtol=1e-5, atol=1e-5)
        o_ref, lse_ref = _oracle_rows(q, ck, cv, rk, rv, npy(pos), m, W, d)
        assert_close(out, o_ref, kind, f"call {call} vs oracle")
        np.testing.assert_allclose(npy(lse), lse_ref, rtol=1e-4, atol=1e-4)


def test_noalloc_lowers_the_split_count_to_fit_its_scratch():
    # a request of 64 splits (33 partial slots per row of 65 key tiles) needs 17.4 MB of
    # partials; the call halves the request until they fit its 16 MiB (32: 22 slots per row,
    # 11.6 MB) and must then agree with hca_attend given that request, and with the oracle
    import long_context_sparse_28_b300 as L
    B, H, d, m, W, Ncap = 16, 64, 128, 128, 128, 8192
    g = torch.Generator().manual_seed(5)
    mk = lambda *s, std=1.0: (torch.randn(*s, generator=g) * std).to(torch.bfloat16).cuda()  # noqa: E731
    ck, cv, rk, rv = mk(B, Ncap, d), mk(B, Ncap, d), mk(B, W, d), mk(B, W, d)
    q = mk(B, 1, H, d, std=d ** -0.5)
    pos = torch.tensor([m * Ncap - 1 - 997 * b for b in range(B)], dtype=torch.int64, device="cuda")
    assert L.hca_attend_workspace(B, 1, H, d, Ncap, W, 64) > L.hca_attend_noalloc_scratch_bytes()
    assert L.hca_attend_workspace(B, 1, H, d, Ncap, W, 32) <= L.hca_attend_noalloc_scratch_bytes()
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, 1, H), float("nan"), device="cuda")
    L.hca_attend_noalloc(q, d ** -0.5, ck, cv, m, rk, rv, W, pos, out, lse, splits=64)
    ref = torch.empty_like(q)
    ref_lse = torch.empty_like(lse)
    L.hca_attend(q, d ** -0.5, ck, cv, m, rk, rv, W, pos, ref, ref_lse, splits=32)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    np.testing.assert_array_equal(npy(out), npy(ref))              # same plan, same arithmetic
    np.testing.assert_array_equal(npy(lse), npy(ref_lse))
    rows = [0, 7, 15]
    o_ref, lse_ref = _oracle_rows(q[rows], ck[rows], cv[rows], rk[rows], rv[rows], npy(pos)[rows], m, W, d)
    assert_close(out[rows], o_ref, "bf16", "lowered split vs oracle")
    np.testing.assert_allclose(npy(lse[rows]), lse_ref, rtol=1e-4, atol=1e-4)


def test_noalloc_rejects_problems_larger_than_its_scratch():
    import long_context_sparse_28_b300 as L
    lib = L.library()
    cap = int(lib.hca_attend_noalloc_scratch_bytes())
    assert cap == 16 << 20
    H, d = 64, 128
    T = cap // (H * (d + 1) * 4) + 1                          # one split per query no longer fits
    q = torch.zeros(1, 1, H, d, dtype=torch.bfloat16, device="cuda")
    ck = torch.zeros(1, 4, d, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(T, dtype=torch.int64, device="cuda")
    P = ctypes.c_void_p
    st = lib.hca_attend_noalloc(P(q.data_ptr()), 1, T, H, d, 0.1, P(ck.data_ptr()), P(ck.data_ptr()), 4, 128,
                                None, None, 0, 0, None, None, None, 0, P(pos.data_ptr()), 0, 1, P(q.data_ptr()),
                                None, None)
    assert st == 6                                           # CSAHCA_ERR_WORKSPACE: refused, nothing enqueued
