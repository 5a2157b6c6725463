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
