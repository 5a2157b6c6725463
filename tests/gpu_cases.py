"""Shared helpers of the GPU parity tests: tolerance checks and whole-workload cases that run
the CUDA path (through the C-ABI binding) and the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as wl

# Tolerances (from the acceptance criteria of the method's specification):
BF16_MAX_ABS, BF16_REL_L2 = 2e-2, 1e-2     # bf16 outputs
F32_MAX_ABS = 1e-4                         # fp32 outputs
TIE_REL = 1e-3                             # index sets may differ only on near-ties of the k-th score


def bf16_half_ulp(r):
    """Half the bfloat16 grid spacing at |r| (the rounding every bf16 output carries)."""
    a = np.abs(np.asarray(r, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 8)


def npy(t):
    return wl.to_numpy(t)


def f64(a):
    return oracle.to_f64(np.asarray(a))


def assert_close(gpu, ref, dtype: str, what=""):
    g = f64(npy(gpu) if torch.is_tensor(gpu) else gpu)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite GPU values"
    if not g.size:
        return 0.0
    if dtype == "f32":
        err = np.abs(g - r).max()
        assert err <= F32_MAX_ABS, f"{what}: max-abs {err:.3e} > {F32_MAX_ABS}"
    else:
        # max-abs 2e-2, literally wherever a bf16 value can meet it; where |o| >= 8 half the bf16
        # grid spacing alone exceeds 2e-2, and there the bound applies to the error beyond the
        # output's own rounding.  Plus the relative L2 bound on the whole tensor.
        hu = bf16_half_ulp(r)
        err = np.maximum(np.abs(g - r) - np.where(hu > BF16_MAX_ABS, hu, 0.0), 0.0).max()
        rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
        assert err <= BF16_MAX_ABS and rel <= BF16_REL_L2, f"{what}: excess max-abs {err:.3e}, rel-L2 {rel:.3e}"
    return err


def check_index_set(gpu_row, ora_row, ora_scores, n_vis: int, k: int, what=""):
    """GPU index row: ascending, -1 padded, min(k, n_vis) distinct visible entries, and equal to
    the oracle's except on entries whose oracle score is within TIE_REL of the k-th score."""
    g = np.asarray(gpu_row, dtype=np.int64)
    o = np.asarray(ora_row, dtype=np.int64)
    take = min(k, n_vis)
    assert (g[take:] == -1).all(), f"{what}: padding"
    gs = g[:take]
    assert (gs >= 0).all() and (gs < n_vis).all(), f"{what}: out-of-range index"
    assert (np.diff(gs) > 0).all(), f"{what}: not strictly ascending"
    diff = set(gs.tolist()) ^ set(o[:take].tolist())
    if diff:
        s = np.asarray(ora_scores[:n_vis], dtype=np.float64)
        kth = np.sort(s)[::-1][take - 1]
        for e in diff:
            assert abs(s[e] - kth) <= TIE_REL * abs(kth), f"{what}: entry {e} score {s[e]} vs k-th {kth}"
    return len(diff)


# ---------------------------------------------------------------------------- decode cases
def csa_decode_case(w: wl.Workload, check_seqs, device="cuda", layer="csa", step_kwargs=None):
    """Builds a CSA decode problem on the GPU (caches from the raw context, then one decode
    step through the C-ABI) and the oracle's answer for the sequences in ``check_seqs``."""
    import long_context_sparse_28_b300 as L
    from long_context_sparse_28_b300.layers import CSACache, CSADecode
    lengths = w.lengths()
    B, m = w.B, w.m_csa
    Ncap = max(lengths) // m + 1
    dtype = wl.torch_dtype(w.kv)
    fmt = L.KEY_FMT[w.key_fmt]
    cache = CSACache(B, Ncap, w.d, w.W, w.d_I, fmt, dtype, device, m=m, kv_fp8=w.kv_cache == "fp8")
    bias = wl.layer_bias(w, layer, m, device)
    k_new = torch.empty(B, 1, w.d, dtype=dtype, device=device)
    v_new = torch.empty_like(k_new)
    g_new = torch.empty(B, 1, dtype=torch.float32, device=device)
    kdt = torch.float32 if w.key_fmt == "f32" else torch.bfloat16
    kidx_new = torch.empty(B, 1, w.d_I, dtype=kdt, device=device)
    host = {}
    for b in range(B):
        Lb = lengths[b]
        k, v, g = wl.raw_tokens(w, layer, b, Lb, device)
        kin = wl.index_key_inputs(w, layer, b, Lb // m + 1, device)
        cache.build_seq(b, k, v, g, bias, kin, Lb - 1)
        k_new[b, 0], v_new[b, 0], g_new[b, 0] = k[Lb - 1], v[Lb - 1], g[Lb - 1]
        kidx_new[b, 0] = kin[(Lb - 1) // m]
        if b in check_seqs:
            host[b] = dict(K=npy(k), V=npy(v), G=npy(g), kin=npy(kin), L=Lb)
        del k, v, g, kin
    q = torch.cat([wl.queries(w, layer, b, 1, device) for b in range(B)])[:, None]
    qi, ww = zip(*[wl.indexer_queries(w, layer, b, 1, device) for b in range(B)])
    q_idx = torch.cat(qi)[:, None]
    wts = torch.cat(ww)[:, None]
    pos = torch.tensor([Lb - 1 for Lb in lengths], dtype=torch.int64, device=device)
    step = CSADecode(cache, w.H, w.H_I, w.k, bias, **(step_kwargs or {}))
    scores = torch.full((B, 1, cache.Ncap), float("nan"), dtype=torch.float32, device=device)
    out, lse, idx = step.step(pos, q, q_idx, wts, k_new, v_new, g_new, kidx_new, scores_out=scores)
    torch.cuda.synchronize()
    st = L.device_status()
    return dict(w=w, cache=cache, step=step, out=out, lse=lse, idx=idx, scores=scores, host=host, q=q,
                q_idx=q_idx, wts=wts, bias=bias, lengths=lengths, status=st, fmt=fmt)


def oracle_csa_seq(case, b, idx_override=None):
    w = case["w"]
    h = case["host"][b]
    Lb, m = h["L"], w.m_csa
    N = Lb // m
    if w.kv_cache == "fp8":                  # FP8 caches: attention reads the dequantised entries
        c8 = oracle.compress_kv_fp8(h["K"], h["V"], h["G"], npy(case["bias"]), m, n_blocks=N)
        ck, cv = c8["ck"], c8["cv"]
        case.setdefault("kv8", {})[b] = c8
    else:
        sd = oracle.BF16 if w.kv == "bf16" else oracle.F32
        ck, cv = oracle.compress(h["K"], h["V"], h["G"], npy(case["bias"]), m, sd, n_blocks=N)
    codes, scales = oracle.quantize_keys(h["kin"][:N], case["fmt"])
    res = oracle.csa_queries(npy(case["q"][b]), npy(case["q_idx"][b]), npy(case["wts"][b]), [Lb - 1], ck, cv,
                             codes, scales, case["fmt"], h["K"], h["V"], 0, m, w.k, w.W, w.scale,
                             idx_override=idx_override)
    return res, ck, cv, codes, scales


def hca_decode_case(w: wl.Workload, check_seqs, device="cuda", layer="hca", splits=0):
    import long_context_sparse_28_b300 as L
    from long_context_sparse_28_b300.layers import HCACache, HCADecode
    lengths = w.lengths()
    B, m = w.B, w.m_hca
    Ncap = max(lengths) // m + 1
    dtype = wl.torch_dtype(w.kv)
    cache = HCACache(B, Ncap, w.d, w.W, dtype, device, m=m, kv_fp8=w.kv_cache == "fp8")
    bias = wl.layer_bias(w, layer, m, device)
    k_new = torch.empty(B, 1, w.d, dtype=dtype, device=device)
    v_new = torch.empty_like(k_new)
    g_new = torch.empty(B, 1, dtype=torch.float32, device=device)
    host = {}
    for b in range(B):
        Lb = lengths[b]
        k, v, g = wl.raw_tokens(w, layer, b, Lb, device)
        cache.build_seq(b, k, v, g, bias, Lb - 1)
        k_new[b, 0], v_new[b, 0], g_new[b, 0] = k[Lb - 1], v[Lb - 1], g[Lb - 1]
        if b in check_seqs:
            host[b] = dict(K=npy(k), V=npy(v), G=npy(g), L=Lb)
        del k, v, g
    q = torch.cat([wl.queries(w, layer, b, 1, device) for b in range(B)])[:, None]
    pos = torch.tensor([Lb - 1 for Lb in lengths], dtype=torch.int64, device=device)
    step = HCADecode(cache, w.H, bias, splits=splits)
    out, lse = step.step(pos, q, k_new, v_new, g_new)
    torch.cuda.synchronize()
    return dict(w=w, cache=cache, step=step, out=out, lse=lse, host=host, q=q, bias=bias, lengths=lengths,
                status=L.device_status())


def oracle_hca_seq(case, b):
    w = case["w"]
    h = case["host"][b]
    Lb, m = h["L"], w.m_hca
    if w.kv_cache == "fp8":
        c8 = oracle.compress_kv_fp8(h["K"], h["V"], h["G"], npy(case["bias"]), m, n_blocks=Lb // m)
        ck, cv = c8["ck"], c8["cv"]
        case.setdefault("kv8", {})[b] = c8
    else:
        sd = oracle.BF16 if w.kv == "bf16" else oracle.F32
        ck, cv = oracle.compress(h["K"], h["V"], h["G"], npy(case["bias"]), m, sd, n_blocks=Lb // m)
    res = oracle.hca_queries(npy(case["q"][b]), [Lb - 1], ck, cv, h["K"], h["V"], 0, m, w.W, w.scale)
    return res, ck, cv


# ----------------------------------------------------------- FP8 compressed K/V (pogovet.com detail 5)
def kv8_planes(ck, cv):
    """GPU FP8 caches [N, 224] / [N, 128] uint8 -> the oracle's planes (K codes, scales, RoPE bf16
    bits; V codes, scales -- the V scales travel in the K row), after checking the zero bytes."""
    k = npy(ck).astype(np.uint8)
    v = npy(cv).astype(np.uint8)
    assert k.shape[1] == 224 and v.shape[1] == 128 and not k[:, 67:96].any(), "layout / padding bytes"
    return dict(k_codes=k[:, :64], k_scales=k[:, 64:65], k_rope=np.ascontiguousarray(k[:, 96:224]).view(np.uint16),
                v_codes=v[:, :128], v_scales=np.ascontiguousarray(k[:, 65:67]))


def kv8_dequant(pl, d=128):
    return (oracle.dequant_kv_fp8(pl["k_codes"], pl["k_scales"], pl["k_rope"], d),
            oracle.dequant_kv_fp8(pl["v_codes"], pl["v_scales"], None, d))


def e4m3_step(deq, scale_bytes, block=64):
    """One E4M3 grid step at each dequantised value, at its block's scale."""
    e = np.repeat(scale_bytes.astype(np.int64) - 127, block, axis=1)[:, : deq.shape[1]]
    z = np.abs(deq) * np.ldexp(1.0, -e)
    k = np.floor(np.log2(np.maximum(z, 2.0 ** -6))).astype(np.int64)
    return np.ldexp(1.0, np.where(z < 2.0 ** -6, -9, k - 3) + e)


def assert_kv8_close(ck, cv, ora, what=""):
    """Pooled FP8 caches against the oracle's (compress_kv_fp8): the pooled float32 values of the
    device and the oracle's fp64 ones rounded to float32 may differ in their last bits, so a code
    may sit one E4M3 step (and a scale one binade) away; the RoPE dims within one bf16 step."""
    g = kv8_planes(ck, cv)
    gk, gv = kv8_dequant(g)
    for name, gd, od, gs, os_ in (("K", gk[:, :64], ora["ck"][:, :64], g["k_scales"], ora["k_scales"]),
                                  ("V", gv, ora["cv"], g["v_scales"], ora["v_scales"])):
        tol = np.maximum(e4m3_step(gd, gs), e4m3_step(od, os_)) + 1e-4   # (+ the pooling's cancellation error)
        assert (np.abs(gd - od) <= tol).all(), f"{what} {name}: beyond one E4M3 step"
        assert np.mean(gs == os_) >= 0.99, f"{what} {name}: scale bytes"
        assert np.abs(gs.astype(int) - os_.astype(int)).max() <= 1, f"{what} {name}: scale off by more than 1"
    assert np.mean(g["k_codes"] == ora["k_codes"]) >= 0.95 and np.mean(g["v_codes"] == ora["v_codes"]) >= 0.95
    # one bf16 step, plus the fp32 pooling's own error where the pooled value cancels (inputs of
    # magnitude <= ~4, up to 128 terms: below 1e-4)
    hu = 2 * bf16_half_ulp(ora["ck"][:, 64:]) + 1e-4
    assert (np.abs(gk[:, 64:] - ora["ck"][:, 64:]) <= hu).all(), f"{what}: RoPE dims"
