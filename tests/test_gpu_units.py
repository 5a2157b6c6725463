"""GPU parity of each hot-path step against the CPU oracle, at sizes the oracle finishes in
seconds that still span several tiles and ragged tails.  All calls go through the C-ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_cases import assert_close, check_index_set, npy

pytestmark = pytest.mark.gpu

L = None


@pytest.fixture(scope="module", autouse=True)
def lib():
    global L
    import long_context_sparse_28_b300 as mod
    L = mod
    torch.manual_seed(0)
    yield mod


def dev_i64(x):
    return torch.tensor(x, dtype=torch.int64, device="cuda")


def rnd(shape, dtype, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(dtype).cuda()


DT = {"f32": torch.float32, "bf16": torch.bfloat16}
SD = {"f32": oracle.F32, "bf16": oracle.BF16}
OKEY = {"f32": oracle.KEY_F32, "bf16": oracle.KEY_BF16, "e4m3": oracle.KEY_E4M3, "e2m1": oracle.KEY_E2M1}


# ------------------------------------------------------------------------ a1/a2 pooling
@pytest.mark.parametrize("m,dt,d", [(1, "f32", 64), (4, "f32", 64), (4, "bf16", 128), (128, "bf16", 128),
                                    (7, "f32", 64), (128, "f32", 64)])
def test_compress_parity_ragged(m, dt, d):
    B, stride = 3, 1000
    k = rnd((B, stride, d), DT[dt], 1)
    v = rnd((B, stride, d), DT[dt], 2)
    g = rnd((B, stride), torch.float32, 3)
    bias = rnd((m,), torch.float32, 4, 0.5)
    pos0 = [0, 2 * m, 3]
    nraw = [stride, 5 * m + 3, 2 * m]
    Ncap = (stride + 3) // m + 2
    ck = torch.full((B, Ncap, d), 7.0, dtype=DT[dt], device="cuda")
    cv = torch.full_like(ck, 7.0)
    L.csa_compress(k, v, g, dev_i64(pos0), dev_i64(nraw), bias, m, ck, cv)
    assert L.device_status() == 0
    for b in range(B):
        j0 = -(-pos0[b] // m)
        j1 = (pos0[b] + nraw[b]) // m
        rows0 = j0 * m - pos0[b]
        nb = max(0, j1 - j0)
        K, V, G = npy(k[b]), npy(v[b]), npy(g[b])
        if nb:
            ok, _ = oracle.pool(np.ascontiguousarray(K[rows0:rows0 + nb * m]), G[rows0:rows0 + nb * m], npy(bias), m)
            ov, _ = oracle.pool(np.ascontiguousarray(V[rows0:rows0 + nb * m]), G[rows0:rows0 + nb * m], npy(bias), m)
            tol = "f32" if dt == "f32" else "bf16"
            assert_close(ck[b, j0:j1], ok, tol, f"ck b={b}")
            assert_close(cv[b, j0:j1], ov, tol, f"cv b={b}")
            if dt == "bf16":   # at most one bf16 ulp from the oracle's once-rounded value
                ref = oracle.bf16_to_f64(oracle.round_bf16(ok))
                got = oracle.to_f64(npy(ck[b, j0:j1]))
                assert (np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30).all()
        untouched = [j for j in range(Ncap) if not (j0 <= j < j1)]
        assert (oracle.to_f64(npy(ck[b, untouched])) == 7.0).all()


# ------------------------------------------------------------------ a4 key quantisation
@pytest.mark.parametrize("fmt", ["f32", "bf16", "e4m3", "e2m1"])
@pytest.mark.parametrize("in_dt", ["f32", "bf16"])
def test_index_key_quantize_bitexact(fmt, in_dt):
    if fmt == "f32" and in_dt == "bf16":
        pytest.skip("fp32 keys come from fp32 inputs")
    rows, d_I = 517, 64
    x = rnd((rows, d_I), torch.float32, 11)
    x[5] = 0.0
    x[6, :32] = 0.0
    x[7] *= 1e-30
    x[8] *= 3e4
    x[9, 3] = 300.0
    x[10, 40] = -5e3
    x[11] = -0.0
    x = x.to(DT[in_dt])
    F = L.KEY_FMT[fmt]
    codes, scales = L.key_storage(1, rows, d_I, F)
    L.csa_index_key_quantize(x, F, codes[0], None if scales is None else scales[0])
    torch.cuda.synchronize()
    if fmt == "bf16" and in_dt == "f32":
        oc, os_ = oracle.round_bf16(oracle.to_f64(npy(x))), None
    else:
        oc, os_ = oracle.quantize_keys(npy(x), OKEY[fmt])
    got = npy(codes[0])
    if fmt == "f32":
        np.testing.assert_array_equal(got.view(np.uint32), np.asarray(oc).view(np.uint32))
    else:
        np.testing.assert_array_equal(got.view(np.uint8).ravel(), np.asarray(oc).view(np.uint8).ravel())
    if os_ is not None:
        np.testing.assert_array_equal(npy(scales[0]).view(np.uint8).ravel(), np.asarray(os_).view(np.uint8).ravel())


# --------------------------------------------------------------------------- a6 top-k
@pytest.mark.parametrize("k", [1, 64, 1024])
def test_topk_from_scores_bitexact(k):
    rng = np.random.default_rng(k)
    N = 5000
    R = 9
    S = rng.standard_normal((R, N)).astype(np.float32)
    S[1] = np.round(S[1] * 3) / 3                       # heavy ties
    S[2] = 1.5                                          # all equal
    S[3, ::2] = 0.0
    S[3, 1::2] = -0.0                                   # signed zeros tie
    S[4] = np.abs(S[4]) * 1e-38                         # subnormals
    S[5] = -np.abs(S[5])
    nv = np.array([N, N, N, N, N, N, k - 1 if k > 1 else 0, k, 0], dtype=np.int64)
    idx = torch.empty(R, k, dtype=torch.int32, device="cuda")
    L.csa_topk_from_scores(torch.from_numpy(S).cuda(), dev_i64(nv), k, idx)
    ref = oracle.topk(S.astype(np.float64), nv, k)
    np.testing.assert_array_equal(npy(idx), ref)


def test_topk_from_scores_long_rows():
    rng = np.random.default_rng(7)
    R, N, k = 3, 262144, 1024
    S = (np.abs(rng.standard_normal((R, N))) * 8).astype(np.float32)
    S[1] = np.round(S[1])                               # coarse scores -> huge boundary bin
    nv = np.array([N, 200000, 1500], dtype=np.int64)
    idx = torch.empty(R, k, dtype=torch.int32, device="cuda")
    L.csa_topk_from_scores(torch.from_numpy(S).cuda(), dev_i64(nv), k, idx)
    np.testing.assert_array_equal(npy(idx), oracle.topk(S.astype(np.float64), nv, k))


@pytest.mark.parametrize("k", [5000, 9000])
def test_topk_from_scores_k_above_4096(k):
    # k = 9000 exceeds the candidate list (8192), so the exact finish runs on whole rows
    rng = np.random.default_rng(k)
    R, N = 4, 40000
    S = rng.standard_normal((R, N)).astype(np.float32)
    S[1] = np.round(S[1] * 2) / 2                       # heavy ties at the boundary
    nv = np.array([N, 30001, k - 3, k], dtype=np.int64)
    idx = torch.empty(R, k, dtype=torch.int32, device="cuda")
    L.csa_topk_from_scores(torch.from_numpy(S).cuda(), dev_i64(nv), k, idx)
    np.testing.assert_array_equal(npy(idx), oracle.topk(S.astype(np.float64), nv, k))


# ---------------------------------------------------------------- bounded device waits
def test_bounded_wait_times_out_and_context_survives():
    # a device wait that nothing completes gives up after its limit, reports a timeout through
    # the error word, and leaves the context usable
    torch.cuda.synchronize()
    assert L.device_status() == 0
    L.selftest_bounded_wait(2_000_000)
    assert L.device_status() == 4                       # CSAHCA_ERR_TIMEOUT
    assert L.device_status() == 0                       # read and cleared
    S = torch.arange(64, dtype=torch.float32, device="cuda")[None]
    idx = torch.empty(1, 8, dtype=torch.int32, device="cuda")
    L.csa_topk_from_scores(S, dev_i64([64]), 8, idx)
    assert L.device_status() == 0
    np.testing.assert_array_equal(npy(idx)[0], np.arange(56, 64))


# ------------------------------------------------------------------- a5 indexer scores
@pytest.mark.parametrize("fmt,q_dt,Ncap,H_I", [("f32", "f32", 700, 16), ("bf16", "bf16", 700, 16),
                                               ("e4m3", "bf16", 700, 16), ("e2m1", "bf16", 700, 16),
                                               ("e4m3", "bf16", 1000, 16), ("e2m1", "bf16", 1000, 16),
                                               ("e2m1", "bf16", 1024, 16), ("e2m1", "bf16", 1024, 32),
                                               ("e2m1", "bf16", 1280, 64), ("e4m3", "bf16", 1000, 64)])
def test_index_scores_and_topk_parity(fmt, q_dt, Ncap, H_I):
    # the tensor-core indexer runs for e4m3 keys with Ncap % 8 == 0 (1000) and e2m1 keys with
    # Ncap % 256 == 0 (1024, 1280); the other cases take the generic kernel
    B, T, d_I, m, k = 2, 3, 64, 4, 96
    F = L.KEY_FMT[fmt]
    kin = rnd((B, Ncap, d_I), torch.float32, 21)
    kin[0, 17] *= 4
    kin = kin.to(torch.float32 if fmt == "f32" else torch.bfloat16)
    codes, scales = L.key_storage(B, Ncap, d_I, F)
    L.csa_index_key_quantize(kin, F, codes, scales)
    q = rnd((B, T, H_I, d_I), DT[q_dt], 22, 0.125)
    w = torch.rand(B, T, H_I, generator=torch.Generator().manual_seed(23)).cuda()
    pos = dev_i64([[4 * Ncap - 1, 1000, 30], [400, 2, 4 * Ncap + 50]])
    idx = torch.empty(B, T, k, dtype=torch.int32, device="cuda")
    sc = torch.full((B, T, Ncap), float("nan"), device="cuda")
    L.csa_index_topk(q, w, codes, scales, F, pos.reshape(-1), m, k, idx, scores_out=sc)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    for b in range(B):
        oc, os_ = oracle.quantize_keys(npy(kin[b]), OKEY[fmt])
        khat = oracle.dequant_keys(F, oc, os_, d_I)
        p = npy(pos[b])
        nv = np.minimum(Ncap, (p + 1) // m)
        S = oracle.index_scores(npy(q[b]), npy(w[b]), khat, nv)
        ref = oracle.topk(S, nv, k)
        for t in range(T):
            got = npy(sc[b, t])[: nv[t]].astype(np.float64)
            scale = np.abs(S[t, : nv[t]]).max() if nv[t] else 1.0
            assert np.abs(got - S[t, : nv[t]]).max(initial=0) <= 1e-5 * scale + 1e-6
            check_index_set(npy(idx[b, t]), ref[t], S[t], int(nv[t]), k, f"b{b}t{t}")


@pytest.mark.parametrize("H_I", [16, 32, 64])
def test_index_fp4_queries_parity(H_I):
    # both indexer operands in FP4: the queries quantised to MX E2M1 (bit-exact with the oracle's
    # rule), then scores against the oracle's scores of the dequantised queries, and the top-k
    B, T, Ncap, d_I, m, k = 3, 2, 5120, 64, 4, 300
    kin = rnd((B, Ncap, d_I), torch.bfloat16, 51)
    kin[1, 7] *= 4
    codes, scales = L.key_storage(B, Ncap, d_I, L.E2M1_UE8M0)
    L.csa_index_key_quantize(kin, L.E2M1_UE8M0, codes, scales)
    q = rnd((B, T, H_I, d_I), torch.bfloat16, 52, 0.125)
    q[0, 1, 3] *= 64                                    # a head with a much larger scale
    q[2, 0, 5, :32] = 0                                 # an all-zero run of 32
    qc = torch.empty(B, T, H_I, d_I // 2, dtype=torch.uint8, device="cuda")
    qs = torch.empty(B, T, H_I, d_I // 32, dtype=torch.uint8, device="cuda")
    L.csa_index_key_quantize(q, L.E2M1_UE8M0, qc, qs)
    w = torch.rand(B, T, H_I, generator=torch.Generator().manual_seed(53)).cuda()
    pos = dev_i64([[4 * Ncap - 1, 3000], [40, 4 * Ncap + 9], [9999, 17]])
    idx = torch.empty(B, T, k, dtype=torch.int32, device="cuda")
    sc = torch.full((B, T, Ncap), float("nan"), device="cuda")
    L.csa_index_topk_fp4(qc, qs, w, codes, scales, pos.reshape(-1), m, k, idx, scores_out=sc)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    for b in range(B):
        oc, os_ = oracle.quantize_keys(npy(q[b]).reshape(T * H_I, d_I), oracle.KEY_E2M1)
        np.testing.assert_array_equal(npy(qc[b]).reshape(T * H_I, -1), oc)
        np.testing.assert_array_equal(npy(qs[b]).reshape(T * H_I, -1), os_)
        kc, ks = oracle.quantize_keys(npy(kin[b]), oracle.KEY_E2M1)
        khat = oracle.dequant_keys(oracle.KEY_E2M1, kc, ks, d_I)
        nv = np.minimum(Ncap, (npy(pos[b]) + 1) // m)
        S = oracle.index_scores(oracle.fp4_query(npy(q[b])), npy(w[b]), khat, nv)
        ref = oracle.topk(S, nv, k)
        for t in range(T):
            got = npy(sc[b, t])[: nv[t]].astype(np.float64)
            assert np.abs(got - S[t, : nv[t]]).max() <= 1e-5 * np.abs(S[t, : nv[t]]).max() + 1e-6
            check_index_set(npy(idx[b, t]), ref[t], S[t], int(nv[t]), k, f"b{b}t{t}")


@pytest.mark.parametrize("H_I", [16, 64])
def test_index_fp4_queries_prefill_form(H_I):
    # more than 256 query rows with the FP4 workspace: keys and queries expanded to bf16 in the
    # workspace (exact), scored by the prefill indexer, top-k with its own histogram; scores and
    # index sets against the oracle's FP4 rule
    from torch.profiler import ProfilerActivity, profile
    B, T, Ncap, d_I, m, k = 1, 320, 2048, 64, 4, 150
    kin = rnd((B, Ncap, d_I), torch.bfloat16, 61)
    kin[0, 11] *= 16
    codes, scales = L.key_storage(B, Ncap, d_I, L.E2M1_UE8M0)
    L.csa_index_key_quantize(kin, L.E2M1_UE8M0, codes, scales)
    q = rnd((B, T, H_I, d_I), torch.bfloat16, 62, 0.125)
    q[0, 5, 1] *= 64
    qc = torch.empty(B, T, H_I, d_I // 2, dtype=torch.uint8, device="cuda")
    qs = torch.empty(B, T, H_I, d_I // 32, dtype=torch.uint8, device="cuda")
    L.csa_index_key_quantize(q, L.E2M1_UE8M0, qc, qs)
    w = torch.rand(B, T, H_I, generator=torch.Generator().manual_seed(63)).cuda()
    pos_np = np.arange(4 * Ncap - 1 - 23 * (T - 1), 4 * Ncap, 23)          # visibility grows along the rows
    pos = dev_i64(pos_np)
    idx = torch.empty(B, T, k, dtype=torch.int32, device="cuda")
    sc = torch.full((B, T, Ncap), float("nan"), device="cuda")
    ws = torch.zeros(L.csa_index_topk_fp4_workspace(B, T, H_I, Ncap, k), dtype=torch.uint8, device="cuda")
    assert ws.numel() > L.csa_index_topk_workspace(B, T, Ncap, k)          # the form applies
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        L.csa_index_topk_fp4(qc, qs, w, codes, scales, pos, m, k, idx, scores_out=sc, workspace=ws)
        torch.cuda.synchronize()
    names = " ".join(e.name for e in prof.events())
    assert "expand_e2m1_rows_kernel" in names and "index_prefill_kernel" in names
    assert L.device_status() == 0
    kc, ks = oracle.quantize_keys(npy(kin[0]), oracle.KEY_E2M1)
    khat = oracle.dequant_keys(oracle.KEY_E2M1, kc, ks, d_I)
    nv = np.minimum(Ncap, (pos_np + 1) // m)
    S = oracle.index_scores(oracle.fp4_query(npy(q[0])), npy(w[0]), khat, nv)
    ref = oracle.topk(S, nv, k)
    for t in range(0, T, 7):
        got = npy(sc[0, t])[: nv[t]].astype(np.float64)
        assert np.abs(got - S[t, : nv[t]]).max() <= 1e-5 * np.abs(S[t, : nv[t]]).max() + 1e-6
        check_index_set(npy(idx[0, t]), ref[t], S[t], int(nv[t]), k, f"t{t}")


@pytest.mark.parametrize("H_I,T", [(16, 24), (32, 12), (64, 6)])
def test_prefill_indexer_tensor_core_parity(H_I, T):
    # bf16 keys and queries with T a multiple of 128 / H_I: the tensor-core prefill kernel (query
    # rows x heads as one MMA operand); rows straddle several 8192-key chunks and a ragged tail
    from torch.profiler import ProfilerActivity, profile
    B, Ncap, d_I, m, k = 2, 20000, 64, 4, 200
    kin = rnd((B, Ncap, d_I), torch.bfloat16, 41)
    codes, _ = L.key_storage(B, Ncap, d_I, L.BF16)
    L.csa_index_key_quantize(kin, L.BF16, codes)
    q = rnd((B, T, H_I, d_I), torch.bfloat16, 42, 0.125)
    w = torch.rand(B, T, H_I, generator=torch.Generator().manual_seed(43)).cuda()
    p0 = [4 * Ncap - T + 3, 4 * 8192 - 5]
    pos = dev_i64([[p0[b] + t for t in range(T)] for b in range(B)])
    idx = torch.empty(B, T, k, dtype=torch.int32, device="cuda")
    sc = torch.full((B, T, Ncap), float("nan"), device="cuda")
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        L.csa_index_topk(q, w, codes, None, L.BF16, pos.reshape(-1), m, k, idx, scores_out=sc)
        torch.cuda.synchronize()
    names = [e.name for e in prof.events()]
    assert any("index_prefill_kernel" in n for n in names), "tensor-core prefill kernel not used"
    assert not any("index_score_kernel" in n for n in names)
    assert L.device_status() == 0
    for b in range(B):
        khat = oracle.dequant_keys(oracle.KEY_BF16, npy(kin[b]), None, d_I)
        nv = np.minimum(Ncap, (npy(pos[b]) + 1) // m)
        S = oracle.index_scores(npy(q[b]), npy(w[b]), khat, nv)
        ref = oracle.topk(S, nv, k)
        for t in range(T):
            got = npy(sc[b, t])[: nv[t]].astype(np.float64)
            assert np.abs(got - S[t, : nv[t]]).max() <= 1e-5 * np.abs(S[t, : nv[t]]).max() + 1e-6
            assert np.isnan(npy(sc[b, t])[nv[t]:]).all()         # entries a row does not see: untouched
            check_index_set(npy(idx[b, t]), ref[t], S[t], int(nv[t]), k, f"b{b}t{t}")


@pytest.mark.parametrize("fmt", ["e2m1", "e4m3"])
def test_index_topk_one_bin_over_65536_keys_per_cta(fmt):
    # 80 rows of 250112 identical index keys: all scores of a row are equal, so the exact top-k
    # is the first k entries (ties to the lower index) and every key of a row lands in one
    # histogram bin.  The tensor-core indexer's CTAs then stream more than 65536 keys of one row
    # each, which its 16-bit shared-memory counts only survive by being flushed in between.
    B, Ncap, d_I, H_I, m, k = 80, 250112, 64, 16, 4, 1024
    F = L.KEY_FMT[fmt]
    one = rnd((1, 8, d_I), torch.bfloat16, 31)
    c1, s1 = L.key_storage(1, 8, d_I, F)
    L.csa_index_key_quantize(one, F, c1, s1)
    codes, scales = L.key_storage(B, Ncap, d_I, F)
    codes.copy_(c1[:, :1].expand_as(codes))
    scales.copy_(s1[:, :1].expand_as(scales))
    q = rnd((B, 1, H_I, d_I), torch.bfloat16, 32, 0.125)
    w = torch.rand(B, 1, H_I, generator=torch.Generator().manual_seed(33)).cuda()
    pos = dev_i64([m * Ncap - 1] * B)
    idx = torch.empty(B, 1, k, dtype=torch.int32, device="cuda")
    L.csa_index_topk(q, w, codes, scales, F, pos, m, k, idx)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    np.testing.assert_array_equal(npy(idx).reshape(B, k), np.broadcast_to(np.arange(k, dtype=np.int32), (B, k)))


# ------------------------------------------------------------------------ a7/a8 attention
def _rand_cache(B, Ncap, W, d, dt, seed):
    ck = rnd((B, Ncap, d), DT[dt], seed)
    cv = rnd((B, Ncap, d), DT[dt], seed + 1)
    rk = rnd((B, W, d), DT[dt], seed + 2)
    rv = rnd((B, W, d), DT[dt], seed + 3)
    return ck, cv, rk, rv


@pytest.mark.parametrize("dt,H,d", [("f32", 8, 64), ("bf16", 64, 128), ("bf16", 32, 128), ("bf16", 16, 128),
                                    ("bf16", 8, 64)])
def test_csa_attend_parity(dt, H, d):
    B, Ncap, W, k = 3, 300, 128, 70
    ck, cv, rk, rv = _rand_cache(B, Ncap, W, d, dt, 30)
    q = rnd((B, 1, H, d), DT[dt], 35, d ** -0.5)
    rng = np.random.default_rng(1)
    idx = np.full((B, 1, k), -1, dtype=np.int32)
    idx[0, 0] = np.sort(rng.choice(Ncap, k, replace=False))
    idx[1, 0, :10] = np.arange(10) * 3                     # mostly padding
    pos = np.array([5000, 1199, 40])                         # seq 2: window reaches before token 0
    out = torch.empty(B, 1, H, d, dtype=DT[dt], device="cuda")
    lse = torch.empty(B, 1, H, device="cuda")
    L.csa_attend(q, d ** -0.5, ck, cv, torch.from_numpy(idx).cuda(), rk, rv, W, dev_i64(pos), out, lse)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    for b in range(B):
        sel = idx[b, 0][idx[b, 0] >= 0]
        wp = np.arange(max(0, pos[b] - W + 1), pos[b] + 1) % W
        o, ls = oracle.attend(npy(q[b, 0]), d ** -0.5, npy(ck[b]), npy(cv[b]), sel, npy(rk[b]), npy(rv[b]), wp)
        assert_close(out[b, 0], o, dt, f"csa b{b}")
        np.testing.assert_allclose(npy(lse[b, 0]), ls, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("splits", [0, 1, 3, 17])
@pytest.mark.parametrize("dt,H,d", [("f32", 8, 64), ("bf16", 64, 128), ("bf16", 32, 128)])
def test_hca_attend_parity(splits, dt, H, d):
    B, m, W = 3, 128, 128
    pos = np.array([128 * 40 + 5, 127, 300])                 # 40 entries; 1 entry; 2 entries
    Ncap = 45
    ck, cv, rk, rv = _rand_cache(B, Ncap, W, d, dt, 40)
    q = rnd((B, 1, H, d), DT[dt], 45, d ** -0.5)
    out = torch.empty(B, 1, H, d, dtype=DT[dt], device="cuda")
    lse = torch.empty(B, 1, H, device="cuda")
    L.hca_attend(q, d ** -0.5, ck, cv, m, rk, rv, W, dev_i64(pos), out, lse, splits=splits)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    for b in range(B):
        nv = min(Ncap, (pos[b] + 1) // m)
        wp = np.arange(max(0, pos[b] - W + 1), pos[b] + 1) % W
        o, ls = oracle.attend(npy(q[b, 0]), d ** -0.5, npy(ck[b]), npy(cv[b]), np.arange(nv), npy(rk[b]),
                              npy(rv[b]), wp)
        assert_close(out[b, 0], o, dt, f"hca b{b}")
        np.testing.assert_allclose(npy(lse[b, 0]), ls, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("B", [48, 140])
def test_attend_piece_schedule_more_rows_than_a_warp(B):
    # 33..256 decode rows take the shared-memory form of the piece schedule (HCA: rows of
    # different lengths; CSA: the host-made schedule with more rows than a warp)
    H, d, m, W, Ncap, k = 64, 128, 128, 128, 45, 200
    rng = np.random.default_rng(B)
    ck, cv, rk, rv = _rand_cache(B, Ncap, W, d, "bf16", 60)
    q = rnd((B, 1, H, d), torch.bfloat16, 61, d ** -0.5)
    pos = rng.integers(0, m * Ncap + 64, size=B)
    pos[0], pos[1] = 5, m * (Ncap + 3)                       # window only; every entry visible
    out = torch.empty(B, 1, H, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, 1, H, device="cuda")
    L.hca_attend(q, d ** -0.5, ck, cv, m, rk, rv, W, dev_i64(pos), out, lse)
    idx = np.full((B, 1, k), -1, dtype=np.int32)
    for b in range(B):                                       # distinct entries, -1 padded
        n = int(rng.integers(0, Ncap + 1))
        idx[b, 0, :n] = np.sort(rng.choice(Ncap, n, replace=False))
    out_c = torch.empty_like(out)
    lse_c = torch.empty_like(lse)
    L.csa_attend(q, d ** -0.5, ck, cv, torch.from_numpy(idx).cuda(), rk, rv, W, dev_i64(pos), out_c, lse_c)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    for b in range(B):
        wp = np.arange(max(0, pos[b] - W + 1), pos[b] + 1) % W
        nv = min(Ncap, (pos[b] + 1) // m)
        o, ls = oracle.attend(npy(q[b, 0]), d ** -0.5, npy(ck[b]), npy(cv[b]), np.arange(nv), npy(rk[b]),
                              npy(rv[b]), wp)
        assert_close(out[b, 0], o, "bf16", f"hca b{b}")
        np.testing.assert_allclose(npy(lse[b, 0]), ls, rtol=1e-5, atol=1e-5)
        sel = idx[b, 0][idx[b, 0] >= 0]
        o, ls = oracle.attend(npy(q[b, 0]), d ** -0.5, npy(ck[b]), npy(cv[b]), sel, npy(rk[b]), npy(rv[b]), wp)
        assert_close(out_c[b, 0], o, "bf16", f"csa b{b}")
        np.testing.assert_allclose(npy(lse_c[b, 0]), ls, rtol=1e-5, atol=1e-5)


def test_attend_empty_key_set_gives_zero():
    B, H, d, Ncap = 1, 8, 64, 4
    ck, cv, rk, rv = _rand_cache(B, Ncap, 1, d, "f32", 50)
    q = rnd((B, 1, H, d), torch.float32, 51)
    idx = torch.full((B, 1, 3), -1, dtype=torch.int32, device="cuda")
    out = torch.full((B, 1, H, d), 9.0, device="cuda")
    lse = torch.zeros(B, 1, H, device="cuda")
    L.csa_attend(q, 0.125, ck, cv, idx, rk, rv, 0, dev_i64([10]), out, lse)
    torch.cuda.synchronize()
    assert (npy(out) == 0).all() and np.isneginf(npy(lse)).all()


def test_attend_window_from_chunk_and_ring():
    # chunked prefill: window tokens >= chunk start come from the chunk, older ones from the ring
    B, H, d, W, T, Ncap = 1, 64, 128, 128, 300, 64
    pos0 = 1024
    ck, cv, rk, rv = _rand_cache(B, Ncap, W, d, "bf16", 60)
    chunk_k = rnd((B, T, d), torch.bfloat16, 61)
    chunk_v = rnd((B, T, d), torch.bfloat16, 62)
    q = rnd((B, T, H, d), torch.bfloat16, 63, d ** -0.5)
    qpos = np.arange(T) + pos0
    out = torch.empty(B, T, H, d, dtype=torch.bfloat16, device="cuda")
    L.hca_attend(q, d ** -0.5, ck, cv, 128, rk, rv, W, dev_i64(qpos), out, None, chunk_k=chunk_k, chunk_v=chunk_v,
                 chunk_pos0=dev_i64([pos0]))
    torch.cuda.synchronize()
    assert L.device_status() == 0
    allk = np.concatenate([npy(rk[0]), npy(chunk_k[0])])      # rows: ring slot s, then chunk
    allv = np.concatenate([npy(rv[0]), npy(chunk_v[0])])
    for t in [0, 1, 127, 128, 200, 299]:
        p = pos0 + t
        toks = np.arange(max(0, p - W + 1), p + 1)
        rows = np.where(toks >= pos0, W + toks - pos0, toks % W)
        nv = min(Ncap, (p + 1) // 128)
        o, _ = oracle.attend(npy(q[0, t]), d ** -0.5, npy(ck[0]), npy(cv[0]), np.arange(nv), allk, allv, rows)
        assert_close(out[0, t], o, "bf16", f"t={t}")


def test_out_of_range_index_is_flagged_not_read():
    B, H, d, Ncap, W = 1, 8, 64, 16, 8
    ck, cv, rk, rv = _rand_cache(B, Ncap, W, d, "f32", 70)
    q = rnd((B, 1, H, d), torch.float32, 71)
    idx = torch.tensor([[[0, 3, Ncap + 5]]], dtype=torch.int32, device="cuda")
    out = torch.empty(B, 1, H, d, device="cuda")
    L.csa_attend(q, 0.125, ck, cv, idx, rk, rv, W, dev_i64([100]), out, None)
    assert L.device_status() == 5          # CSAHCA_ERR_BOUNDS
    assert L.device_status() == 0          # cleared
    o, _ = oracle.attend(npy(q[0, 0]), 0.125, npy(ck[0]), npy(cv[0]), [0, 3], npy(rk[0]), npy(rv[0]),
                         np.arange(93, 101) % W)
    assert_close(out[0, 0], o, "f32", "skipped entry")


# ----------------------------------------------------------------------- a3 cache append
@pytest.mark.parametrize("m,fmt", [(4, "e2m1"), (4, "e4m3"), (128, None)])
def test_append_tokenwise_and_chunked_match_bulk(m, fmt):
    B, d, W, d_I = 2, 128, 128, 64
    Ltot = 3 * m + 5 + 600
    k = rnd((B, Ltot, d), torch.bfloat16, 80)
    v = rnd((B, Ltot, d), torch.bfloat16, 81)
    g = rnd((B, Ltot), torch.float32, 82)
    kin = rnd((B, Ltot // m + 2, d_I), torch.bfloat16, 83)
    bias = rnd((m,), torch.float32, 84, 0.5)
    Ncap = Ltot // m + 1
    F = L.KEY_FMT[fmt] if fmt else None
    ck = torch.zeros(B, Ncap, d, dtype=torch.bfloat16, device="cuda")
    cv = torch.zeros_like(ck)
    rk = torch.zeros(B, W, d, dtype=torch.bfloat16, device="cuda")
    rv = torch.zeros_like(rk)
    rg = torch.zeros(B, W, device="cuda")
    codes, scales = L.key_storage(B, Ncap, d_I, F) if fmt else (None, None)
    # phase 1: tokens one at a time; phase 2: one chunk of 600 tokens at an unaligned position
    n1 = 3 * m + 5
    for t in range(n1):
        pos = dev_i64([t, t])
        j = t // m
        if fmt:
            L.csa_cache_append(k[:, t:t + 1].contiguous(), v[:, t:t + 1].contiguous(), g[:, t:t + 1].contiguous(),
                               kin[:, j:j + 1].contiguous(), pos, bias, m, rk, rv, rg, ck, cv, codes, scales, F)
        else:
            L.hca_cache_append(k[:, t:t + 1].contiguous(), v[:, t:t + 1].contiguous(), g[:, t:t + 1].contiguous(),
                               pos, bias, m, rk, rv, rg, ck, cv)
    n2 = 600
    j0 = n1 // m
    pos = dev_i64([n1, n1])
    if fmt:
        L.csa_cache_append(k[:, n1:].contiguous(), v[:, n1:].contiguous(), g[:, n1:].contiguous(),
                           kin[:, j0:j0 + n2 // m + 1].contiguous(), pos, bias, m, rk, rv, rg, ck, cv, codes, scales, F)
    else:
        L.hca_cache_append(k[:, n1:].contiguous(), v[:, n1:].contiguous(), g[:, n1:].contiguous(), pos, bias, m,
                           rk, rv, rg, ck, cv)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    nb = Ltot // m
    for b in range(B):
        ok, ov = oracle.compress(npy(k[b]), npy(v[b]), npy(g[b]), npy(bias), m, oracle.BF16, n_blocks=nb)
        assert_close(ck[b, :nb], oracle.bf16_to_f64(ok), "bf16", "append ck")
        assert_close(cv[b, :nb], oracle.bf16_to_f64(ov), "bf16", "append cv")
        # the ring holds the last W tokens
        slots = np.arange(Ltot - W, Ltot) % W
        np.testing.assert_array_equal(npy(rk[b])[slots], npy(k[b])[Ltot - W:])
        np.testing.assert_array_equal(npy(rg[b])[slots], npy(g[b])[Ltot - W:])
        if fmt:
            oc, os_ = oracle.quantize_keys(npy(kin[b])[:nb], OKEY[fmt])
            np.testing.assert_array_equal(npy(codes[b, :nb]).view(np.uint8), np.asarray(oc).view(np.uint8))
            np.testing.assert_array_equal(npy(scales[b, :nb]).view(np.uint8), np.asarray(os_).view(np.uint8))


def test_decode_step_is_deterministic():
    from tests.gpu_cases import csa_decode_case
    w = wl.shrink(wl.WORKLOADS["csa_decode_b8_128k_bf16"], B=2, L=(5003, 4100))
    a = csa_decode_case(w, [])
    out1, idx1 = a["out"].clone(), a["idx"].clone()
    b = csa_decode_case(w, [])
    assert torch.equal(out1, b["out"]) and torch.equal(idx1, b["idx"])


def test_attend_tensor_core_row_without_keys_gives_zero():
    # bf16, H = 64: a row with no visible entry and no window (W = 0) is written by the CTA the
    # schedule gives it (o = 0, lse = -inf); the other row is merged by its last CTA
    B, H, d, m, Ncap = 2, 64, 128, 128, 8
    ck, cv, _, _ = _rand_cache(B, Ncap, 1, d, "bf16", 52)
    q = rnd((B, 1, H, d), torch.bfloat16, 53, d ** -0.5)
    pos = np.array([5, 128 * 3 + 1])
    out = torch.full((B, 1, H, d), 9.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, 1, H, device="cuda")
    L.hca_attend(q, d ** -0.5, ck, cv, m, None, None, 0, dev_i64(pos), out, lse, splits=2)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    assert (npy(out[0]) == 0).all() and np.isneginf(npy(lse[0])).all()
    o, ls = oracle.attend(npy(q[1, 0]), d ** -0.5, npy(ck[1]), npy(cv[1]), np.arange(3), None, None, [])
    assert_close(out[1, 0], o, "bf16", "row with keys")
    np.testing.assert_allclose(npy(lse[1, 0]), ls, rtol=1e-5, atol=1e-5)


def test_attend_many_rows_one_split_written_directly():
    # more rows than the piece schedule takes and one split per row: every row is one item whose
    # CTA writes the bf16 output and lse itself (no partials, no merge launch); rows without keys
    # (no complete block, W = 0) give o = 0, lse = -inf
    B, H, d, m, Ncap = 300, 64, 128, 128, 8
    ck, cv, _, _ = _rand_cache(B, Ncap, 1, d, "bf16", 54)
    q = rnd((B, 1, H, d), torch.bfloat16, 55, d ** -0.5)
    rng = np.random.default_rng(56)
    pos = rng.integers(0, m * Ncap, size=B)
    pos[::7] = rng.integers(0, m - 1, size=len(pos[::7]))      # no complete block yet
    out = torch.full((B, 1, H, d), 9.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, 1, H, device="cuda")
    L.hca_attend(q, d ** -0.5, ck, cv, m, None, None, 0, dev_i64(pos), out, lse)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    o_g, l_g = npy(out), npy(lse)
    for b in range(B):
        n = (int(pos[b]) + 1) // m
        if n == 0:
            assert (o_g[b] == 0).all() and np.isneginf(l_g[b]).all(), b
            continue
        o, ls = oracle.attend(npy(q[b, 0]), d ** -0.5, npy(ck[b]), npy(cv[b]), np.arange(n), None, None, [])
        assert_close(out[b, 0], o, "bf16", f"row {b}")
        np.testing.assert_allclose(l_g[b, 0], ls, rtol=1e-5, atol=1e-5)


def test_workspace_state_is_cleared_by_every_call():
    # the top-k's per-row histograms and the attention's per-row arrival counters live in the
    # caller's workspace: after each call they are zero again, so calls on one workspace give the
    # results of calls on fresh ones
    B, T, Ncap, d_I, H_I, m, k = 3, 2, 1024, 64, 16, 4, 100
    F = L.KEY_FMT["e2m1"]
    R = B * T
    ws = torch.zeros(L.csa_index_topk_workspace(B, T, Ncap, k), dtype=torch.uint8, device="cuda")
    ins = []
    for s in range(2):
        kin = rnd((B, Ncap, d_I), torch.bfloat16, 70 + s)
        codes, scales = L.key_storage(B, Ncap, d_I, F)
        L.csa_index_key_quantize(kin, F, codes, scales)
        q = rnd((B, T, H_I, d_I), torch.bfloat16, 72 + s, 0.125)
        w = torch.rand(B, T, H_I, generator=torch.Generator().manual_seed(74 + s)).cuda()
        pos = dev_i64([4 * Ncap - 1 - 37 * i for i in range(R)])
        ins.append((q, w, codes, scales, pos))

    def topk(i, wsp):
        q, w, codes, scales, pos = ins[i]
        idx = torch.empty(B, T, k, dtype=torch.int32, device="cuda")
        L.csa_index_topk(q, w, codes, scales, F, pos, m, k, idx, workspace=wsp)
        return idx

    a1, b1, a2 = topk(0, ws), topk(1, ws), topk(0, ws)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    assert not ws[: R * 4096 * 4].any(), "histograms left behind"
    fresh = torch.zeros_like(ws)
    assert torch.equal(a1, a2) and torch.equal(b1, topk(1, fresh))
    # attention: the same workspace for an HCA and a CSA call, twice
    H, d, W, Nc = 64, 128, 128, 60
    ck, cv, rk, rv = _rand_cache(B, Nc, W, d, "bf16", 80)
    qa = rnd((B, 1, H, d), torch.bfloat16, 81, d ** -0.5)
    pa = dev_i64([128 * 50 + 3, 128 * 7, 900])
    sel = torch.arange(k, dtype=torch.int32, device="cuda").remainder(Nc).reshape(1, 1, k).repeat(B, 1, 1)
    wsa = torch.zeros(max(L.hca_attend_workspace(B, 1, H, d, Nc, W), L.csa_attend_workspace(B, 1, H, d, k, W)),
                      dtype=torch.uint8, device="cuda")

    def att(wsp):
        oh, lh = torch.empty_like(qa), torch.empty(B, 1, H, device="cuda")
        oc, lc = torch.empty_like(qa), torch.empty(B, 1, H, device="cuda")
        L.hca_attend(qa, d ** -0.5, ck, cv, 128, rk, rv, W, pa, oh, lh, workspace=wsp)
        L.csa_attend(qa, d ** -0.5, ck, cv, sel, rk, rv, W, pa, oc, lc, workspace=wsp)
        return oh, lh, oc, lc

    r1, r2, r3 = att(wsa), att(wsa), att(torch.zeros_like(wsa))
    torch.cuda.synchronize()
    assert L.device_status() == 0
    assert not wsa[: 65536 * 4].any(), "arrival counters left behind"
    for x, y, z in zip(r1, r2, r3):
        assert torch.equal(x, y) and torch.equal(x, z)
