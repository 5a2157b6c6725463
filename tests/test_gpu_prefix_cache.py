"""On-disk prefix caches on the GPU: a CSA and an HCA layer state saved after a prefix, restored
into a slot of a running batch, then one decode step through the C-ABI; the restored slot's
outputs must match the oracle computed from the prefix's raw tokens plus the new token
(honbul.tistory.com/221, "KV cache를 줄이는 방식": the compressed cache of a shared prefix is
stored and reused)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_cases import assert_close, check_index_set, npy

pytestmark = pytest.mark.gpu


def test_restored_prefix_decodes_like_the_oracle(tmp_path):
    import long_context_sparse_28_b300 as L
    from long_context_sparse_28_b300 import cache_io
    from long_context_sparse_28_b300.layers import CSACache, CSADecode, HCACache, HCADecode
    dev = "cuda"
    w = wl.shrink(wl.WORKLOADS["decode_1m_b32_csa_hca"], B=3, L_range=(), L=(6000, 9001, 4500), k=256)
    Ls = w.lengths()
    n_ctx = Ls[1] - 1                                    # the prefix; its next token is at n_ctx
    Ncap_c, Ncap_h = max(Ls) // 4 + 8, max(Ls) // 128 + 1
    cb, hb = wl.layer_bias(w, "csa", 4, dev), wl.layer_bias(w, "hca", 128, dev)
    raw = {}
    # ---- the prefix alone (one sequence), saved to disk
    src_c = CSACache(1, Ncap_c, w.d, w.W, w.d_I, L.E2M1_UE8M0, torch.bfloat16, dev)
    src_h = HCACache(1, Ncap_h, w.d, w.W, torch.bfloat16, dev)
    k, v, g = wl.raw_tokens(w, "csa", 1, Ls[1], dev)
    kin = wl.index_key_inputs(w, "csa", 1, Ls[1] // 4 + 1, dev)
    hk, hv, hg = wl.raw_tokens(w, "hca", 1, Ls[1], dev)
    src_c.build_seq(0, k, v, g, cb, kin, n_ctx)
    src_h.build_seq(0, hk, hv, hg, hb, n_ctx)
    raw[1] = (k, v, g, kin, hk, hv, hg)
    cache_io.save_prefix(str(tmp_path / "c.kv"), src_c, [n_ctx])
    cache_io.save_prefix(str(tmp_path / "h.kv"), src_h, [n_ctx])
    del src_c, src_h
    # ---- a running batch: slots 0 and 2 built from their own tokens, slot 1 restored
    csa = CSACache(3, Ncap_c, w.d, w.W, w.d_I, L.E2M1_UE8M0, torch.bfloat16, dev)
    hca = HCACache(3, Ncap_h, w.d, w.W, torch.bfloat16, dev)
    for b in (0, 2):
        k, v, g = wl.raw_tokens(w, "csa", b, Ls[b], dev)
        kin = wl.index_key_inputs(w, "csa", b, Ls[b] // 4 + 1, dev)
        hk, hv, hg = wl.raw_tokens(w, "hca", b, Ls[b], dev)
        csa.build_seq(b, k, v, g, cb, kin, Ls[b] - 1)
        hca.build_seq(b, hk, hv, hg, hb, Ls[b] - 1)
        raw[b] = (k, v, g, kin, hk, hv, hg)
    csa.ck[1].fill_(7.0)                                 # stale contents the restore must replace
    hca.ck[1].fill_(7.0)
    assert cache_io.load_prefix_into(str(tmp_path / "c.kv"), csa, 1) == n_ctx
    assert cache_io.load_prefix_into(str(tmp_path / "h.kv"), hca, 1) == n_ctx
    # ---- one decode step for the batch
    st = lambda i: torch.stack([raw[b][i][Ls[b] - 1] for b in range(3)])[:, None].contiguous()  # noqa: E731
    kidx_new = torch.stack([raw[b][3][(Ls[b] - 1) // 4] for b in range(3)])[:, None].contiguous()
    q = torch.cat([wl.queries(w, "csa", b, 1, dev) for b in range(3)])[:, None]
    qh = torch.cat([wl.queries(w, "hca", b, 1, dev) for b in range(3)])[:, None]
    qi, ww = zip(*[wl.indexer_queries(w, "csa", b, 1, dev) for b in range(3)])
    q_idx, wts = torch.cat(qi)[:, None], torch.cat(ww)[:, None]
    pos = torch.tensor([Lb - 1 for Lb in Ls], dtype=torch.int64, device=dev)
    scores = torch.full((3, 1, csa.Ncap), float("nan"), device=dev)
    out_c, lse_c, idx = CSADecode(csa, w.H, w.H_I, w.k, cb).step(pos, q, q_idx, wts, st(0), st(1), st(2)[..., 0],
                                                                  kidx_new, scores_out=scores)
    out_h, lse_h = HCADecode(hca, w.H, hb).step(pos, qh, st(4), st(5), st(6)[..., 0])
    torch.cuda.synchronize()
    assert L.device_status() == 0
    # ---- the oracle on the restored sequence's raw tokens (prefix + the new token)
    for b in (1, 0):
        K, V, G, KIN, HK, HV, HG = (npy(t) for t in raw[b])
        Lb = Ls[b]
        N = Lb // 4
        ck, cv = oracle.compress(K, V, G, npy(cb), 4, oracle.BF16)
        codes, sc = oracle.quantize_keys(KIN[:N], oracle.KEY_E2M1)
        res = oracle.csa_queries(npy(q[b]), npy(q_idx[b]), npy(wts[b]), [Lb - 1], ck, cv, codes, sc,
                                 oracle.KEY_E2M1, K, V, 0, 4, w.k, w.W, w.scale)
        check_index_set(npy(idx[b, 0]), res["idx"][0], res["scores"][0], N, w.k, f"slot {b}")
        res2 = oracle.csa_queries(npy(q[b]), npy(q_idx[b]), npy(wts[b]), [Lb - 1], ck, cv, codes, sc,
                                  oracle.KEY_E2M1, K, V, 0, 4, w.k, w.W, w.scale, idx_override=npy(idx[b]))
        assert_close(out_c[b, 0], res2["o"][0], "bf16", f"CSA slot {b}")
        np.testing.assert_allclose(npy(lse_c[b, 0]), res2["lse"][0], rtol=1e-4, atol=1e-4)
        hck, hcv = oracle.compress(HK, HV, HG, npy(hb), 128, oracle.BF16)
        hres = oracle.hca_queries(npy(qh[b]), [Lb - 1], hck, hcv, HK, HV, 0, 128, w.W, w.scale)
        assert_close(out_h[b, 0], hres["o"][0], "bf16", f"HCA slot {b}")
        np.testing.assert_allclose(npy(lse_h[b, 0]), hres["lse"][0], rtol=1e-4, atol=1e-4)
