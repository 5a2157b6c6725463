"""End-to-end GPU parity on the five synthetic workloads, at their full sizes and in the launch
configuration the benchmark times; the oracle computes the sampled sequences / query rows
one by one from the same seeded raw inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_cases import (assert_close, assert_kv8_close, check_index_set, csa_decode_case, hca_decode_case, npy,
                             oracle_csa_seq, oracle_hca_seq)

pytestmark = pytest.mark.gpu


def _check_csa(case, seqs, tol):
    w = case["w"]
    assert case["status"] == 0
    for b in seqs:
        res, ck, cv, codes, scales = oracle_csa_seq(case, b)
        Lb = case["lengths"][b]
        N = Lb // w.m_csa
        # compressed cache: within one storage ulp (FP8: one E4M3 step) of the oracle's
        if w.kv_cache == "fp8":
            assert_kv8_close(case["cache"].ck[b, :N], case["cache"].cv[b, :N], case["kv8"][b], f"ck b{b}")
        else:
            assert_close(case["cache"].ck[b, :N], oracle.to_f64(ck), tol, f"ck b{b}")
        # index keys: bit-exact
        np.testing.assert_array_equal(npy(case["cache"].k_codes[b, :N]).view(np.uint8),
                                      np.asarray(codes).view(np.uint8))
        # scores and the selected set
        S = res["scores"][0]
        got = npy(case["scores"][b, 0])[:N].astype(np.float64)
        assert np.abs(got - S[:N]).max() <= 1e-5 * np.abs(S[:N]).max() + 1e-6
        check_index_set(npy(case["idx"][b, 0]), res["idx"][0], S, N, w.k, f"seq {b}")
        # attention, evaluated on the GPU's index set
        res2, *_ = oracle_csa_seq(case, b, idx_override=npy(case["idx"][b]))
        assert_close(case["out"][b, 0], res2["o"][0], tol, f"out b{b}")
        np.testing.assert_allclose(npy(case["lse"][b, 0]), res2["lse"][0], rtol=1e-4, atol=1e-4)


def test_tiny_csa_decode_f32():
    w = wl.WORKLOADS["tiny_csa_decode_f32"]
    case = csa_decode_case(w, [0])
    _check_csa(case, [0], "f32")


def test_csa_decode_b8_128k_bf16():
    w = wl.WORKLOADS["csa_decode_b8_128k_bf16"]
    case = csa_decode_case(w, list(range(w.B)))
    _check_csa(case, list(range(w.B)), "bf16")


def _check_hca(case, seqs):
    w = case["w"]
    assert case["status"] == 0
    for b in seqs:
        res, ck, cv = oracle_hca_seq(case, b)
        n = case["lengths"][b] // w.m_hca
        if w.kv_cache == "fp8":
            assert_kv8_close(case["cache"].ck[b, :n], case["cache"].cv[b, :n], case["kv8"][b], f"hca ck b{b}")
        else:
            assert_close(case["cache"].ck[b, :n], oracle.to_f64(ck), "bf16", f"hca ck b{b}")
        assert_close(case["out"][b, 0], res["o"][0], "bf16", f"hca out b{b}")
        np.testing.assert_allclose(npy(case["lse"][b, 0]), res["lse"][0], rtol=1e-4, atol=1e-4)


def test_hca_decode_b4_1m_bf16():
    w = wl.WORKLOADS["hca_decode_b4_1m_bf16"]
    case = hca_decode_case(w, list(range(w.B)))
    _check_hca(case, list(range(w.B)))


def test_decode_1m_b32_csa_then_hca():
    w = wl.WORKLOADS["decode_1m_b32_csa_hca"]
    lens = w.lengths()
    order = np.argsort(lens)
    seqs = sorted({int(order[0]), int(order[len(order) // 3]), int(order[2 * len(order) // 3]), int(order[-1])})
    csa = csa_decode_case(w, seqs, layer="csa")
    _check_csa(csa, seqs, "bf16")
    del csa
    torch.cuda.empty_cache()
    hca = hca_decode_case(w, seqs, layer="hca")
    _check_hca(hca, seqs)


def test_decode_1m_b32_with_fp8_caches():
    # the 1M decode workload with FP8 compressed K/V (the RoPE dims of K in bf16), four sampled
    # sequences through both layers, at full size in the benchmark's launch configuration
    w = wl.WORKLOADS["decode_1m_b32_csa_hca_kv8"]
    lens = w.lengths()
    order = np.argsort(lens)
    seqs = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    csa = csa_decode_case(w, seqs, layer="csa")
    _check_csa(csa, seqs, "bf16")
    del csa
    torch.cuda.empty_cache()
    hca = hca_decode_case(w, seqs, layer="hca")
    _check_hca(hca, seqs)


def test_hybrid_prefill_t4096_at_256k():
    import long_context_sparse_28_b300 as L
    from long_context_sparse_28_b300.layers import CSACache, HCACache, hybrid_prefill_chunk
    w = wl.WORKLOADS["hybrid_prefill_t4096_at_256k_bf16"]
    x = wl.prefill_inputs(w, "cuda")
    o, T, W = w.offset, w.T, w.W
    n_csa, n_hca = o // w.m_csa, o // w.m_hca
    csa = CSACache(1, (o + T) // w.m_csa, w.d, W, w.d_I, L.BF16, torch.bfloat16)
    hca = HCACache(1, (o + T) // w.m_hca, w.d, W, torch.bfloat16)
    csa.ck[0, :n_csa] = x["csa_ck"]
    csa.cv[0, :n_csa] = x["csa_cv"]
    L.csa_index_key_quantize(x["csa_kidx"], L.BF16, csa.k_codes[0, :n_csa])
    hca.ck[0, :n_hca] = x["hca_ck"]
    hca.cv[0, :n_hca] = x["hca_cv"]
    pos_ring = torch.tensor([o - W], dtype=torch.int64, device="cuda")
    for c in (csa, hca):
        L.swa_ring_write(x["ring_k"][None], x["ring_v"][None], x["ring_gate"][None], pos_ring, W, c.ring_k,
                         c.ring_v, c.ring_gate)
    res = hybrid_prefill_chunk(csa, hca, o, T, x["chunk_k"][None], x["chunk_v"][None], x["chunk_gate"][None],
                               x["chunk_kidx"][None], x["q_csa"][None], x["q_idx"][None], x["w"][None],
                               x["q_hca"][None], x["csa_bias"], x["hca_bias"], w.k)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    # oracle state: prior entries + entries pooled from the chunk; raw tokens = ring + chunk
    h = {k: npy(v) for k, v in x.items()}
    cck, ccv = oracle.compress(h["chunk_k"], h["chunk_v"], h["chunk_gate"], h["csa_bias"], w.m_csa, oracle.BF16)
    hck, hcv = oracle.compress(h["chunk_k"], h["chunk_v"], h["chunk_gate"], h["hca_bias"], w.m_hca, oracle.BF16)
    assert_close(csa.ck[0, n_csa:n_csa + T // 4], oracle.to_f64(cck), "bf16", "chunk csa entries")
    assert_close(hca.ck[0, n_hca:n_hca + T // 128], oracle.to_f64(hck), "bf16", "chunk hca entries")
    ck_all = np.concatenate([h["csa_ck"], cck])
    cv_all = np.concatenate([h["csa_cv"], ccv])
    kidx_all = np.concatenate([h["csa_kidx"], h["chunk_kidx"]])
    hk_all = np.concatenate([h["hca_ck"], hck])
    hv_all = np.concatenate([h["hca_cv"], hcv])
    rawk = np.concatenate([h["ring_k"], h["chunk_k"]])
    rawv = np.concatenate([h["ring_v"], h["chunk_v"]])
    rng = np.random.default_rng(0)
    edge = [0, 1, 2, 3, 4, 127, 128, 129, 1023, 2047, 2048, 4095]
    rest = rng.choice(np.setdiff1d(np.arange(T), edge), 256 - len(edge), replace=False)
    rows = np.unique(np.concatenate([edge, rest]))
    assert len(rows) == 256
    pos = o + rows
    ores = oracle.csa_queries(h["q_csa"][rows], h["q_idx"][rows], h["w"][rows], pos, ck_all, cv_all, kidx_all, None,
                              oracle.KEY_BF16, rawk, rawv, o - W, w.m_csa, w.k, W, w.scale)
    gidx = npy(res["idx"][0])
    for i, t in enumerate(rows):
        nv = (pos[i] + 1) // w.m_csa
        check_index_set(gidx[t], ores["idx"][i], ores["scores"][i], nv, w.k, f"row {t}")
    ores2 = oracle.csa_queries(h["q_csa"][rows], h["q_idx"][rows], h["w"][rows], pos, ck_all, cv_all, kidx_all, None,
                               oracle.KEY_BF16, rawk, rawv, o - W, w.m_csa, w.k, W, w.scale,
                               idx_override=gidx[rows])
    assert_close(res["csa_out"][0, rows], ores2["o"], "bf16", "prefill csa out")
    hres = oracle.hca_queries(h["q_hca"][rows], pos, hk_all, hv_all, rawk, rawv, o - W, w.m_hca, W, w.scale)
    assert_close(res["hca_out"][0, rows], hres["o"], "bf16", "prefill hca out")
    np.testing.assert_allclose(npy(res["hca_lse"][0, rows]), hres["lse"], rtol=1e-4, atol=1e-4)
    # the rings now hold the chunk's last W tokens
    slots = np.arange(o + T - W, o + T) % W
    np.testing.assert_array_equal(npy(csa.ring_k[0])[slots], h["chunk_k"][T - W:])


def test_hybrid_prefill_with_fp4_indexer():
    # the prefill chunk with e2m1 index keys and FP4 (MX E2M1) indexer queries: the indexer runs
    # both operands in FP4 on the block-scaled tensor core; 64 sampled query rows against the oracle's
    # FP4-query rule, then CSA attention on the GPU's index sets
    import long_context_sparse_28_b300 as L
    from long_context_sparse_28_b300.layers import CSACache, HCACache, HybridPrefill
    w = wl.WORKLOADS["hybrid_prefill_t4096_at_256k_q4"]
    x = wl.prefill_inputs(w, "cuda")
    o, T, W = w.offset, w.T, w.W
    n_csa, n_hca = o // w.m_csa, o // w.m_hca
    csa = CSACache(1, (o + T) // w.m_csa, w.d, W, w.d_I, L.E2M1_UE8M0, torch.bfloat16)
    hca = HCACache(1, (o + T) // w.m_hca, w.d, W, torch.bfloat16)
    csa.ck[0, :n_csa] = x["csa_ck"]
    csa.cv[0, :n_csa] = x["csa_cv"]
    L.csa_index_key_quantize(x["csa_kidx"], L.E2M1_UE8M0, csa.k_codes[0, :n_csa], csa.k_scale[0, :n_csa])
    hca.ck[0, :n_hca] = x["hca_ck"]
    hca.cv[0, :n_hca] = x["hca_cv"]
    pos_ring = torch.tensor([o - W], dtype=torch.int64, device="cuda")
    for c in (csa, hca):
        L.swa_ring_write(x["ring_k"][None], x["ring_v"][None], x["ring_gate"][None], pos_ring, W, c.ring_k,
                         c.ring_v, c.ring_gate)
    step = HybridPrefill(csa, hca, T, w.H, w.k, x["csa_bias"], x["hca_bias"], H_I=w.H_I, q_fp4=True)
    step.set_position(o)
    res = step.step(x["chunk_k"][None], x["chunk_v"][None], x["chunk_gate"][None], x["chunk_kidx"][None],
                    x["q_csa"][None], x["q_idx"][None], x["w"][None], x["q_hca"][None])
    torch.cuda.synchronize()
    assert L.device_status() == 0
    h = {k: npy(v) for k, v in x.items()}
    cck, ccv = oracle.compress(h["chunk_k"], h["chunk_v"], h["chunk_gate"], h["csa_bias"], w.m_csa, oracle.BF16)
    ck_all = np.concatenate([h["csa_ck"], cck])
    cv_all = np.concatenate([h["csa_cv"], ccv])
    codes, sc = oracle.quantize_keys(np.concatenate([h["csa_kidx"], h["chunk_kidx"]]), oracle.KEY_E2M1)
    np.testing.assert_array_equal(npy(csa.k_codes[0, :len(codes)]), codes)   # the chunk's keys, bit-exact
    rawk = np.concatenate([h["ring_k"], h["chunk_k"]])
    rawv = np.concatenate([h["ring_v"], h["chunk_v"]])
    rng = np.random.default_rng(1)
    edge = [0, 3, 4, 1023, 4095]
    rows = np.unique(np.concatenate([edge, rng.choice(np.setdiff1d(np.arange(T), edge), 64 - len(edge),
                                                      replace=False)]))
    pos = o + rows
    ores = oracle.csa_queries(h["q_csa"][rows], h["q_idx"][rows], h["w"][rows], pos, ck_all, cv_all, codes, sc,
                              oracle.KEY_E2M1, rawk, rawv, o - W, w.m_csa, w.k, W, w.scale, q_fp4=True)
    gidx = npy(res["idx"][0])
    for i, t in enumerate(rows):
        nv = (pos[i] + 1) // w.m_csa
        check_index_set(gidx[t], ores["idx"][i], ores["scores"][i], nv, w.k, f"row {t}")
    ores2 = oracle.csa_queries(h["q_csa"][rows], h["q_idx"][rows], h["w"][rows], pos, ck_all, cv_all, codes, sc,
                               oracle.KEY_E2M1, rawk, rawv, o - W, w.m_csa, w.k, W, w.scale, q_fp4=True,
                               idx_override=gidx[rows])
    assert_close(res["csa_out"][0, rows], ores2["o"], "bf16", "fp4 prefill csa out")
