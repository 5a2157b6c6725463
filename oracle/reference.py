"""Step-by-step compositions of the oracle primitives (test infrastructure only).

These follow the order in which the pages describe the method: compress the KV
stream into blocks (softmax-gated pooling, m=4 for CSA, m=128 for HCA), let the
lightning indexer score each query against every visible compressed entry, keep the
top-k, and attend jointly over the kept entries plus a raw sliding window (CSA); or
attend over every visible compressed entry plus the window (HCA).  Sources:
honbul.tistory.com/221 (sections "CSA", "HCA", "KV cache를 줄이는 방식") and the
pogovet.com DeepSeek-V4 article, detail 4.

Readings taken where the pages are silent (each one is listed in the design notes):
  * positions are 0-based; compressed entry j (tokens j*m .. j*m+m-1) is visible to a
    query at position p iff its last token is <= p, i.e. j < (p+1)//m ("causally
    complete"); ``strict=True`` gives the alternative j < p//m;
  * the window is the W raw tokens max(0, p-W+1) .. p, including the query's own;
  * window rows and compressed rows form one joint softmax, with no de-duplication;
  * all query heads share one KV stream and one top-k set per query.
"""
from __future__ import annotations

import numpy as np

from . import (BF16, F32, attend, dequant_keys, dequant_kv_fp8, fp4_query, index_scores, pool, quant_kv_fp8,
               quantize_keys, round_to, topk)

__all__ = ["n_visible", "window_positions", "compress", "compress_kv_fp8", "csa_queries", "hca_queries"]

D_ROPE = 64   # RoPE dimensions of a K row kept in BF16 under FP8 storage (a reading: the pages give no width)


def n_visible(pos, m: int, n_entries=None, strict: bool = False):
    """Number of compressed entries visible to a query at ``pos``."""
    pos = np.asarray(pos, dtype=np.int64)
    n = (pos // m) if strict else ((pos + 1) // m)
    if n_entries is not None:
        n = np.minimum(n, n_entries)
    return n


def window_positions(pos: int, W: int) -> np.ndarray:
    return np.arange(max(0, pos - W + 1), pos + 1, dtype=np.int64)


def compress(raw_k, raw_v, gate, bias, m: int, store_dtype: int, n_blocks=None):
    """Pool every complete block of m tokens of K and V (shared weights), then round
    once to the storage dtype.  Returns (ck, cv) in storage form."""
    pk, _ = pool(raw_k, gate, bias, m, n_blocks)
    pv, _ = pool(raw_v, gate, bias, m, n_blocks)
    return round_to(pk, store_dtype), round_to(pv, store_dtype)


def compress_kv_fp8(raw_k, raw_v, gate, bias, m: int, n_blocks=None, d_rope: int = D_ROPE):
    """Pool like ``compress``, then store the entries in FP8 with the RoPE dims of K in BF16
    (pogovet.com article, detail 5; ``oc_quant_kv_fp8``).  Returns a dict with the K planes (codes,
    scales, rope), the V planes (codes, scales) and the dequantised caches ck, cv (fp64 [N, d]),
    which attention reads."""
    pk, _ = pool(raw_k, gate, bias, m, n_blocks)
    pv, _ = pool(raw_v, gate, bias, m, n_blocks)
    d = pk.shape[1]
    kc, ks, kr = quant_kv_fp8(pk, d_rope)
    vc, vs, _ = quant_kv_fp8(pv, 0)
    return dict(k_codes=kc, k_scales=ks, k_rope=kr, v_codes=vc, v_scales=vs,
                ck=dequant_kv_fp8(kc, ks, kr, d), cv=dequant_kv_fp8(vc, vs, np.zeros((len(vc), 0), np.uint16), d))


def _window_rows(pos: int, W: int, raw_pos0: int):
    wp = window_positions(pos, W)
    if wp.size:
        assert wp[0] >= raw_pos0, "window reaches before the raw tokens given to the oracle"
    return wp - raw_pos0


def csa_queries(q, q_idx, w, pos, ck, cv, key_codes, key_scales, key_fmt, raw_k, raw_v,
                raw_pos0: int, m: int, k: int, W: int, scale: float, idx_override=None,
                strict: bool = False, q_fp4: bool = False):
    """CSA for T queries of one sequence.

    q: [T, H, d]; q_idx: [T, H_I, d_I]; w: [T, H_I]; pos: [T] query positions;
    ck, cv: compressed cache [N, d] (storage form); key_codes/key_scales/key_fmt: index
    keys of the N entries; raw_k/raw_v: raw tokens from position raw_pos0 on.
    ``idx_override`` ([T, k]) replaces the oracle's own top-k (used to evaluate attention
    on another implementation's index set).  ``q_fp4``: the indexer queries are taken in FP4
    (``fp4_query``) before scoring.
    Returns dict(o [T,H,d], lse [T,H], idx [T,k], scores [T,N]).
    """
    q = np.asarray(q)
    T = q.shape[0]
    N = ck.shape[0]
    pos = np.asarray(pos, dtype=np.int64).reshape(T)
    nv = n_visible(pos, m, N, strict)
    d_I = q_idx.shape[-1]
    khat = dequant_keys(key_fmt, key_codes, key_scales, d_I)
    S = index_scores(fp4_query(q_idx) if q_fp4 else q_idx, w, khat, nv)
    idx = topk(S, nv, k) if idx_override is None else np.asarray(idx_override, dtype=np.int32)
    H, d = q.shape[1], q.shape[2]
    o = np.empty((T, H, d))
    lse = np.empty((T, H))
    for t in range(T):
        sel = idx[t][idx[t] >= 0].astype(np.int64)
        assert (sel < nv[t]).all(), "selected entry not visible"
        o[t], lse[t] = attend(q[t], scale, ck, cv, sel, raw_k, raw_v,
                              _window_rows(int(pos[t]), W, raw_pos0))
    return dict(o=o, lse=lse, idx=idx, scores=S)


def hca_queries(q, pos, ck, cv, raw_k, raw_v, raw_pos0: int, m: int, W: int, scale: float,
                strict: bool = False):
    """HCA for T queries of one sequence: dense over every visible compressed entry plus
    the raw window.  Returns dict(o [T,H,d], lse [T,H])."""
    q = np.asarray(q)
    T, H, d = q.shape
    N = ck.shape[0]
    pos = np.asarray(pos, dtype=np.int64).reshape(T)
    nv = n_visible(pos, m, N, strict)
    o = np.empty((T, H, d))
    lse = np.empty((T, H))
    for t in range(T):
        o[t], lse[t] = attend(q[t], scale, ck, cv, np.arange(nv[t]), raw_k, raw_v,
                              _window_rows(int(pos[t]), W, raw_pos0))
    return dict(o=o, lse=lse)
