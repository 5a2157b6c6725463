"""FP8 compressed K/V with the RoPE dims of K in BF16 (pogovet.com article, detail 5), on the GPU
through the C-ABI: the quantiser bit for bit against the oracle (pooling with m = 1 passes the rows
through unchanged), pooling and appends against the oracle's pooled-then-quantised caches, and
attention over FP8 caches (HCA tiles by TMA, CSA rows gathered) against the oracle's attention on
the dequantised caches."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_cases import assert_close, assert_kv8_close, kv8_dequant, kv8_planes, npy

pytestmark = pytest.mark.gpu
L = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global L
    import long_context_sparse_28_b300 as lib
    lib.library()
    L = lib


def dev_i64(x):
    return torch.tensor(np.asarray(x, dtype=np.int64).reshape(-1), dtype=torch.int64, device="cuda")


def rnd(shape, dtype, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(dtype).cuda()


def test_quantiser_bit_exact():
    # rows of very different magnitudes, zero blocks, exact powers of two, and 448 * 2^e itself
    N, d = 300, 128
    g = torch.Generator().manual_seed(7)
    x = torch.randn(N, d, generator=g) * torch.exp(torch.empty(N, 1).uniform_(-30, 30, generator=g))
    x[3] = 0.0
    x[4, :64] = 0.0
    x[5, 64:] = 0.0
    x[6, 7] = 448.0 * 2.0 ** -5
    x[7] = torch.ldexp(torch.ones(d), torch.arange(d) % 40 - 20)
    xb = x.to(torch.bfloat16).cuda()
    ck = torch.full((1, N, L.KV_FP8_K_ROW), 0xAB, dtype=torch.uint8, device="cuda")
    cv = torch.full((1, N, L.KV_FP8_V_ROW), 0xAB, dtype=torch.uint8, device="cuda")
    gate = torch.zeros(1, N, device="cuda")
    L.csa_compress(xb[None], xb[None], gate, dev_i64([0]), dev_i64([N]), torch.zeros(1, device="cuda"), 1, ck, cv)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    pl = kv8_planes(ck[0], cv[0])
    xo = npy(xb)
    kc, ks, kr = oracle.quant_kv_fp8(xo, 64)
    vc, vs, _ = oracle.quant_kv_fp8(xo, 0)
    np.testing.assert_array_equal(pl["k_codes"], kc)
    np.testing.assert_array_equal(pl["k_scales"], ks)
    np.testing.assert_array_equal(pl["k_rope"], kr)
    np.testing.assert_array_equal(pl["v_codes"], vc)
    np.testing.assert_array_equal(pl["v_scales"], vs)


@pytest.mark.parametrize("m", [4, 128])
def test_pooling_and_appends_against_the_oracle(m):
    B, d, W, d_I = 2, 128, 128, 64
    Ltot = 3 * m + 5 + 600
    k = rnd((B, Ltot, d), torch.bfloat16, 90)
    v = rnd((B, Ltot, d), torch.bfloat16, 91)
    v[:, 17] *= 40.0                                       # one loud token: its block gets a larger scale
    g = rnd((B, Ltot), torch.float32, 92)
    bias = rnd((m,), torch.float32, 93, 0.5)
    Ncap = Ltot // m + 1
    nb = Ltot // m
    # bulk pooling
    ck = torch.zeros(B, Ncap, L.KV_FP8_K_ROW, dtype=torch.uint8, device="cuda")
    cv = torch.zeros(B, Ncap, L.KV_FP8_V_ROW, dtype=torch.uint8, device="cuda")
    L.csa_compress(k, v, g, dev_i64([0] * B), dev_i64([Ltot] * B), bias, m, ck, cv)
    # appends: tokens one at a time, then a chunk of 600 at an unaligned position
    ck2, cv2 = torch.zeros_like(ck), torch.zeros_like(cv)
    rk = torch.zeros(B, W, d, dtype=torch.bfloat16, device="cuda")
    rv, rg = torch.zeros_like(rk), torch.zeros(B, W, device="cuda")
    kin = rnd((B, Ltot // m + 2, d_I), torch.bfloat16, 94)
    codes, scales = L.key_storage(B, Ncap, d_I, L.E2M1_UE8M0)
    n1 = 3 * m + 5
    for t in range(n1):
        j = t // m
        L.csa_cache_append(k[:, t:t + 1].contiguous(), v[:, t:t + 1].contiguous(), g[:, t:t + 1].contiguous(),
                           kin[:, j:j + 1].contiguous(), dev_i64([t] * B), bias, m, rk, rv, rg, ck2, cv2, codes,
                           scales, L.E2M1_UE8M0)
    j0 = n1 // m
    L.csa_cache_append(k[:, n1:].contiguous(), v[:, n1:].contiguous(), g[:, n1:].contiguous(),
                       kin[:, j0:j0 + 600 // m + 1].contiguous(), dev_i64([n1] * B), bias, m, rk, rv, rg, ck2, cv2,
                       codes, scales, L.E2M1_UE8M0)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    for b in range(B):
        ora = oracle.compress_kv_fp8(npy(k[b]), npy(v[b]), npy(g[b]), npy(bias), m, n_blocks=nb)
        assert_kv8_close(ck[b, :nb], cv[b, :nb], ora, f"bulk b{b}")
        assert_kv8_close(ck2[b, :nb], cv2[b, :nb], ora, f"append b{b}")
        slots = np.arange(Ltot - W, Ltot) % W
        np.testing.assert_array_equal(npy(rk[b])[slots], npy(k[b])[Ltot - W:])


def _fp8_cache(B, Ncap, seed, m=4):
    """FP8 caches pooled on the device from seeded raw tokens (all Ncap entries complete)."""
    d = 128
    n = Ncap * m
    k = rnd((B, n, d), torch.bfloat16, seed)
    v = rnd((B, n, d), torch.bfloat16, seed + 1)
    g = rnd((B, n), torch.float32, seed + 2)
    bias = rnd((m,), torch.float32, seed + 3, 0.5)
    ck = torch.zeros(B, Ncap, L.KV_FP8_K_ROW, dtype=torch.uint8, device="cuda")
    cv = torch.zeros(B, Ncap, L.KV_FP8_V_ROW, dtype=torch.uint8, device="cuda")
    L.csa_compress(k, v, g, dev_i64([0] * B), dev_i64([n] * B), bias, m, ck, cv)
    return ck, cv


@pytest.mark.parametrize("H", [64, 32])
@pytest.mark.parametrize("splits", [0, 3])
def test_hca_attention_over_fp8_caches(H, splits):
    B, d, m, W, Ncap = 3, 128, 128, 128, 300
    ck, cv = _fp8_cache(B, Ncap, 100)
    rk = rnd((B, W, d), torch.bfloat16, 110)
    rv = rnd((B, W, d), torch.bfloat16, 111)
    q = rnd((B, 1, H, d), torch.bfloat16, 112, d ** -0.5)
    pos = np.array([128 * 290 + 5, 127, 128 * 40])           # 290 entries; 1 entry; 41 entries
    out = torch.empty(B, 1, H, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, 1, H, device="cuda")
    L.hca_attend(q, d ** -0.5, ck, cv, m, rk, rv, W, dev_i64(pos), out, lse, splits=splits)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    for b in range(B):
        kd, vd = kv8_dequant(kv8_planes(ck[b], cv[b]))
        nv = min(Ncap, (pos[b] + 1) // m)
        wp = np.arange(max(0, pos[b] - W + 1), pos[b] + 1) % W
        o, ls = oracle.attend(npy(q[b, 0]), d ** -0.5, kd, vd, np.arange(nv), npy(rk[b]), npy(rv[b]), wp)
        assert_close(out[b, 0], o, "bf16", f"hca fp8 b{b}")
        np.testing.assert_allclose(npy(lse[b, 0]), ls, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("H", [64, 32])
def test_csa_attention_over_fp8_caches(H):
    B, d, W, Ncap, k = 4, 128, 128, 700, 300
    ck, cv = _fp8_cache(B, Ncap, 120)
    rk = rnd((B, W, d), torch.bfloat16, 130)
    rv = rnd((B, W, d), torch.bfloat16, 131)
    q = rnd((B, 1, H, d), torch.bfloat16, 132, d ** -0.5)
    rng = np.random.default_rng(5)
    pos = np.array([4 * Ncap + 3, 60, 4 * 500, 2 * 128 + 1])
    idx = np.full((B, 1, k), -1, dtype=np.int32)
    for b in range(B):
        nv = min(Ncap, (pos[b] + 1) // 4)
        n = min(nv, k - 13 * b)
        idx[b, 0, :n] = np.sort(rng.choice(nv, n, replace=False))
    out = torch.empty(B, 1, H, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, 1, H, device="cuda")
    L.csa_attend(q, d ** -0.5, ck, cv, torch.from_numpy(idx).cuda(), rk, rv, W, dev_i64(pos), out, lse)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    for b in range(B):
        kd, vd = kv8_dequant(kv8_planes(ck[b], cv[b]))
        sel = idx[b, 0][idx[b, 0] >= 0]
        wp = np.arange(max(0, pos[b] - W + 1), pos[b] + 1) % W
        o, ls = oracle.attend(npy(q[b, 0]), d ** -0.5, kd, vd, sel, npy(rk[b]), npy(rv[b]), wp)
        assert_close(out[b, 0], o, "bf16", f"csa fp8 b{b}")
        np.testing.assert_allclose(npy(lse[b, 0]), ls, rtol=1e-5, atol=1e-5)


def test_fp8_caches_need_the_tensor_core_shape():
    # FP8 caches run on the tensor-core path only (bf16 queries, d = 128, H in {32, 64})
    B, d, Ncap = 1, 128, 8
    ck, cv = _fp8_cache(B, Ncap, 140)
    q = rnd((B, 1, 16, d), torch.bfloat16, 141, d ** -0.5)
    out = torch.empty_like(q)
    with pytest.raises(L.CsaHcaError, match="status 2"):
        L.hca_attend(q, d ** -0.5, ck, cv, 4, None, None, 0, dev_i64([31]), out)
