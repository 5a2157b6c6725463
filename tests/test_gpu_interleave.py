"""The layer-interleave timeline (pogovet.com article, detail 5: the first two layers HCA, then CSA and
HCA alternating, an MTP block with sliding-window attention only): one decode step through a small
stack, captured and replayed as one CUDA graph, every layer's output checked against the oracle
computed from that layer's own raw tokens."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_cases import assert_close, check_index_set, npy

pytestmark = pytest.mark.gpu


def test_interleaved_stack_graph_step_matches_the_oracle():
    import long_context_sparse_28_b300 as L
    from long_context_sparse_28_b300.layers import (CSACache, HCACache, InterleavedDecode, SWACache,
                                                    interleave_kinds)
    dev = "cuda"
    kinds = interleave_kinds(5)
    assert kinds == ["hca", "hca", "csa", "hca", "csa", "swa"]
    w = wl.shrink(wl.WORKLOADS["decode_1m_b32_csa_hca"], B=2, L_range=(), L=(3000, 4100), k=256)
    Ls = w.lengths()
    B = w.B
    caches, biases, raw = [], [], []
    for i, kind in enumerate(kinds):
        tag = f"l{i}"
        if kind == "csa":
            c = CSACache(B, max(Ls) // 4 + 8, w.d, w.W, w.d_I, L.E2M1_UE8M0, torch.bfloat16, dev)
            bias = wl.layer_bias(w, tag, 4, dev)
        elif kind == "hca":
            c = HCACache(B, max(Ls) // 128 + 1, w.d, w.W, torch.bfloat16, dev)
            bias = wl.layer_bias(w, tag, 128, dev)
        else:
            c = SWACache(B, w.d, w.W, torch.bfloat16, dev)
            bias = None
        per = []
        for b, Lb in enumerate(Ls):
            k, v, g = wl.raw_tokens(w, tag, b, Lb, dev)
            if kind == "csa":
                kin = wl.index_key_inputs(w, tag, b, Lb // 4 + 1, dev)
                c.build_seq(b, k, v, g, bias, kin, Lb - 1)
            elif kind == "hca":
                kin = None
                c.build_seq(b, k, v, g, bias, Lb - 1)
            else:
                kin = None
                c.build_seq(b, k, v, g, Lb - 1)
            per.append((k, v, g, kin))
        caches.append(c)
        biases.append(bias)
        raw.append(per)
    stack = InterleavedDecode(kinds, caches, w.H, w.H_I, w.k, biases)
    pos = torch.tensor([Lb - 1 for Lb in Ls], dtype=torch.int64, device=dev)
    inputs = []
    for i, kind in enumerate(kinds):
        tag = f"l{i}"
        per = raw[i]
        x = {"q": torch.cat([wl.queries(w, tag, b, 1, dev) for b in range(B)])[:, None],
             "k_new": torch.stack([per[b][0][Ls[b] - 1] for b in range(B)])[:, None].contiguous(),
             "v_new": torch.stack([per[b][1][Ls[b] - 1] for b in range(B)])[:, None].contiguous(),
             "gate_new": torch.stack([per[b][2][Ls[b] - 1] for b in range(B)])[:, None].contiguous()}
        if kind == "csa":
            qi, ww = zip(*[wl.indexer_queries(w, tag, b, 1, dev) for b in range(B)])
            x["q_idx"], x["w"] = torch.cat(qi)[:, None], torch.cat(ww)[:, None]
            x["kidx_new"] = torch.stack([per[b][3][(Ls[b] - 1) // 4] for b in range(B)])[:, None].contiguous()
        inputs.append(x)
    # one graph for the whole stack's step (the calls run once outside capture first: per-device set-up)
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            outs = stack.step(pos, inputs)
    g.replay()
    torch.cuda.synchronize()
    assert L.device_status() == 0
    for i, kind in enumerate(kinds):
        o, lse = outs[i]
        for b, Lb in enumerate(Ls):
            K, V, G, KIN = (None if t is None else npy(t) for t in raw[i][b])
            qb = npy(inputs[i]["q"][b])
            if kind == "csa":
                ck, cv = oracle.compress(K, V, G, npy(biases[i]), 4, oracle.BF16)
                codes, sc = oracle.quantize_keys(KIN[: Lb // 4], oracle.KEY_E2M1)
                idx = stack.steps[i].idx
                res = oracle.csa_queries(qb, npy(inputs[i]["q_idx"][b]), npy(inputs[i]["w"][b]), [Lb - 1], ck, cv, codes,
                                         sc, oracle.KEY_E2M1, K, V, 0, 4, w.k, w.W, w.scale)
                check_index_set(npy(idx[b, 0]), res["idx"][0], res["scores"][0], Lb // 4, w.k, f"layer {i} b{b}")
                ref = oracle.csa_queries(qb, npy(inputs[i]["q_idx"][b]), npy(inputs[i]["w"][b]), [Lb - 1], ck, cv,
                                         codes, sc, oracle.KEY_E2M1, K, V, 0, 4, w.k, w.W, w.scale,
                                         idx_override=npy(idx[b]))
            elif kind == "hca":
                hk, hv = oracle.compress(K, V, G, npy(biases[i]), 128, oracle.BF16)
                ref = oracle.hca_queries(qb, [Lb - 1], hk, hv, K, V, 0, 128, w.W, w.scale)
            else:
                rows = oracle.window_positions(Lb - 1, w.W)
                o_, l_ = oracle.attend(qb[0], w.scale, None, None, [], K, V, rows)
                ref = {"o": o_[None], "lse": l_[None]}
            assert_close(o[b, 0], ref["o"][0], "bf16", f"layer {i} ({kind}) b{b}")
            np.testing.assert_allclose(npy(lse[b, 0]), ref["lse"][0], rtol=1e-4, atol=1e-4)
