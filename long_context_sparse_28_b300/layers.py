"""Cache objects and step sequences for a CSA layer and an HCA layer, built only from the
C-ABI entry points (``long_context_sparse_28_b300``).  Torch allocates the buffers; every
operation on their contents is a library kernel.

Cache layout (honbul.tistory.com/221, "KV cache를 줄이는 방식": compressed cache, window cache
and tail state kept apart; not paged):
  ck, cv      [B, Ncap, d]   compressed entries, contiguous per sequence
  ring_k/v    [B, W, d]      the last W raw tokens (token t in slot t % W); it also holds the
  ring_gate   [B, W]         tail of the block being filled (W >= m - 1)
  k_codes     [B, Ncap, ..]  CSA only: lightning-indexer keys in their storage format
  k_scale     [B, Ncap, ..]
"""
from __future__ import annotations

import math

import torch

from . import (BF16, F32, csa_attend, csa_attend_workspace, csa_cache_append, csa_compress, csa_index_key_quantize,
               csa_index_topk, csa_index_topk_workspace, hca_attend, hca_attend_workspace, hca_cache_append,
               hca_compress, key_storage, swa_ring_write)


def _i64(x, device):
    return torch.as_tensor(x, dtype=torch.int64, device=device).reshape(-1).contiguous()


class CSACache:
    """Compressed sparse attention cache of B sequences (m = 4 by default)."""

    def __init__(self, B, Ncap, d, W, d_I, key_fmt, dtype, device="cuda", m=4):
        Ncap = (Ncap + 7) // 8 * 8      # capacity in multiples of 8 entries (tensor-core indexer tiles)
        self.B, self.Ncap, self.d, self.W, self.d_I, self.m = B, Ncap, d, W, d_I, m
        self.key_fmt, self.dtype, self.device = key_fmt, dtype, device
        self.ck = torch.zeros(B, Ncap, d, dtype=dtype, device=device)
        self.cv = torch.zeros(B, Ncap, d, dtype=dtype, device=device)
        self.ring_k = torch.zeros(B, W, d, dtype=dtype, device=device)
        self.ring_v = torch.zeros(B, W, d, dtype=dtype, device=device)
        self.ring_gate = torch.zeros(B, W, dtype=torch.float32, device=device)
        self.k_codes, self.k_scale = key_storage(B, Ncap, d_I, key_fmt, device)
        if self.k_scale is not None:
            self.k_scale.zero_()
        self.k_codes.zero_()

    def build_seq(self, b, k_raw, v_raw, gate, slot_bias, kidx_in, n_ctx):
        """Fills sequence b from its first n_ctx raw tokens: pools every complete block,
        quantises the index keys of those entries and loads the last W tokens into the ring."""
        dev = self.device
        n_blocks = n_ctx // self.m
        csa_compress(k_raw[None, :n_ctx], v_raw[None, :n_ctx], gate[None, :n_ctx], _i64([0], dev),
                     _i64([n_ctx], dev), slot_bias, self.m, self.ck[b:b + 1], self.cv[b:b + 1])
        if n_blocks:
            csa_index_key_quantize(kidx_in[:n_blocks].contiguous(), self.key_fmt, self.k_codes[b, :n_blocks],
                                   None if self.k_scale is None else self.k_scale[b, :n_blocks])
        _fill_ring(self, b, k_raw, v_raw, gate, n_ctx)


class HCACache:
    """Heavily compressed attention cache of B sequences (m = 128 by default)."""

    def __init__(self, B, Ncap, d, W, dtype, device="cuda", m=128):
        self.B, self.Ncap, self.d, self.W, self.m, self.dtype, self.device = B, Ncap, d, W, m, dtype, device
        self.ck = torch.zeros(B, Ncap, d, dtype=dtype, device=device)
        self.cv = torch.zeros(B, Ncap, d, dtype=dtype, device=device)
        self.ring_k = torch.zeros(B, W, d, dtype=dtype, device=device)
        self.ring_v = torch.zeros(B, W, d, dtype=dtype, device=device)
        self.ring_gate = torch.zeros(B, W, dtype=torch.float32, device=device)

    def build_seq(self, b, k_raw, v_raw, gate, slot_bias, n_ctx):
        dev = self.device
        hca_compress(k_raw[None, :n_ctx], v_raw[None, :n_ctx], gate[None, :n_ctx], _i64([0], dev),
                     _i64([n_ctx], dev), slot_bias, self.m, self.ck[b:b + 1], self.cv[b:b + 1])
        _fill_ring(self, b, k_raw, v_raw, gate, n_ctx)


def _fill_ring(c, b, k_raw, v_raw, gate, n_ctx):
    n = min(c.W, n_ctx)
    if n == 0:
        return
    lo = n_ctx - n
    swa_ring_write(k_raw[None, lo:n_ctx].contiguous(), v_raw[None, lo:n_ctx].contiguous(),
                   gate[None, lo:n_ctx].contiguous(), _i64([lo], c.device), n,
                   c.ring_k[b:b + 1], c.ring_v[b:b + 1], c.ring_gate[b:b + 1])


class CSADecode:
    """One CSA decode step for all B sequences: append the new token (pooling a block when it
    completes), score every visible entry with the lightning indexer, keep the top-k, attend
    over them plus the window.  Buffers are preallocated so the step can be graph-captured."""

    def __init__(self, cache: CSACache, H, H_I, k, slot_bias, scale=None):
        self.c, self.H, self.H_I, self.k = cache, H, H_I, k
        self.slot_bias = slot_bias
        B, d, dev = cache.B, cache.d, cache.device
        self.scale = 1.0 / math.sqrt(d) if scale is None else scale
        self.idx = torch.empty(B, 1, k, dtype=torch.int32, device=dev)
        self.out = torch.empty(B, 1, H, d, dtype=cache.dtype, device=dev)
        self.lse = torch.empty(B, 1, H, dtype=torch.float32, device=dev)
        self.ws_topk = torch.empty(csa_index_topk_workspace(B, 1, cache.Ncap, k), dtype=torch.uint8, device=dev)
        self.ws_att = torch.empty(max(256, csa_attend_workspace(B, 1, H, d, k, cache.W)), dtype=torch.uint8,
                                  device=dev)

    def step(self, pos, q, q_idx, w, k_new, v_new, gate_new, kidx_new, scores_out=None):
        """pos int64 [B]: position of the new token (= the query).  q [B,1,H,d]; q_idx [B,1,H_I,d_I];
        w [B,1,H_I]; k_new/v_new [B,1,d]; gate_new [B,1]; kidx_new [B,1,d_I] (used when a block
        completes)."""
        c = self.c
        csa_cache_append(k_new, v_new, gate_new, kidx_new, pos, self.slot_bias, c.m, c.ring_k, c.ring_v,
                         c.ring_gate, c.ck, c.cv, c.k_codes, c.k_scale, c.key_fmt)
        csa_index_topk(q_idx, w, c.k_codes, c.k_scale, c.key_fmt, pos, c.m, self.k, self.idx,
                       scores_out=scores_out, workspace=self.ws_topk)
        csa_attend(q, self.scale, c.ck, c.cv, self.idx, c.ring_k, c.ring_v, c.W, pos, self.out, self.lse,
                   workspace=self.ws_att)
        return self.out, self.lse, self.idx


class HCADecode:
    """One HCA decode step: append (pool when a 128-token block completes) and dense attention
    over every visible entry plus the window."""

    def __init__(self, cache: HCACache, H, slot_bias, scale=None, splits=0):
        self.c, self.H, self.slot_bias, self.splits = cache, H, slot_bias, splits
        B, d, dev = cache.B, cache.d, cache.device
        self.scale = 1.0 / math.sqrt(d) if scale is None else scale
        self.out = torch.empty(B, 1, H, d, dtype=cache.dtype, device=dev)
        self.lse = torch.empty(B, 1, H, dtype=torch.float32, device=dev)
        self.ws = torch.empty(max(256, hca_attend_workspace(B, 1, H, d, cache.Ncap, cache.W, splits)),
                              dtype=torch.uint8, device=dev)

    def step(self, pos, q, k_new, v_new, gate_new):
        c = self.c
        hca_cache_append(k_new, v_new, gate_new, pos, self.slot_bias, c.m, c.ring_k, c.ring_v, c.ring_gate, c.ck,
                         c.cv)
        hca_attend(q, self.scale, c.ck, c.cv, c.m, c.ring_k, c.ring_v, c.W, pos, self.out, self.lse,
                   splits=self.splits, workspace=self.ws)
        return self.out, self.lse


def hybrid_prefill_chunk(csa: CSACache, hca: HCACache, pos0, T, chunk_k, chunk_v, chunk_gate, kidx_chunk,
                         q_csa, q_idx, w, q_hca, csa_bias, hca_bias, k, scale=None, scores_out=None):
    """Chunked prefill of one chunk of T tokens starting at position pos0 (B sequences, same
    pos0): compress the chunk's complete blocks into both caches, quantise the new index keys,
    run CSA (indexer, top-k, sparse attention with the causal window) and HCA (dense, causal)
    for every query of the chunk, then move the chunk's last tokens into both rings.

    chunk_k/v [B, T, d]; chunk_gate [B, T]; kidx_chunk [B, T // m_csa, d_I] (index keys of the
    new CSA entries); q_csa/q_hca [B, T, H, d]; q_idx [B, T, H_I, d_I]; w [B, T, H_I].
    pos0 must be a multiple of both block sizes.  Returns dict of outputs."""
    B, _, d = chunk_k.shape
    dev = csa.device
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    assert pos0 % csa.m == 0 and pos0 % hca.m == 0
    p0 = _i64([pos0] * B, dev)
    nT = _i64([T] * B, dev)
    csa_compress(chunk_k, chunk_v, chunk_gate, p0, nT, csa_bias, csa.m, csa.ck, csa.cv)
    hca_compress(chunk_k, chunk_v, chunk_gate, p0, nT, hca_bias, hca.m, hca.ck, hca.cv)
    j0, nb = pos0 // csa.m, T // csa.m
    for b in range(B):
        csa_index_key_quantize(kidx_chunk[b, :nb].contiguous(), csa.key_fmt, csa.k_codes[b, j0:j0 + nb],
                               None if csa.k_scale is None else csa.k_scale[b, j0:j0 + nb])
    q_pos = (torch.arange(T, device=dev, dtype=torch.int64)[None, :] + pos0).repeat(B, 1).reshape(-1).contiguous()
    H = q_csa.shape[2]
    idx = torch.empty(B, T, k, dtype=torch.int32, device=dev)
    csa_index_topk(q_idx, w, csa.k_codes, csa.k_scale, csa.key_fmt, q_pos, csa.m, k, idx, scores_out=scores_out)
    out_c = torch.empty(B, T, H, d, dtype=csa.dtype, device=dev)
    lse_c = torch.empty(B, T, H, dtype=torch.float32, device=dev)
    csa_attend(q_csa, scale, csa.ck, csa.cv, idx, csa.ring_k, csa.ring_v, csa.W, q_pos, out_c, lse_c,
               chunk_k=chunk_k, chunk_v=chunk_v, chunk_pos0=p0)
    out_h = torch.empty(B, T, H, d, dtype=hca.dtype, device=dev)
    lse_h = torch.empty(B, T, H, dtype=torch.float32, device=dev)
    hca_attend(q_hca, scale, hca.ck, hca.cv, hca.m, hca.ring_k, hca.ring_v, hca.W, q_pos, out_h, lse_h,
               chunk_k=chunk_k, chunk_v=chunk_v, chunk_pos0=p0)
    swa_ring_write(chunk_k, chunk_v, chunk_gate, p0, T, csa.ring_k, csa.ring_v, csa.ring_gate)
    swa_ring_write(chunk_k, chunk_v, chunk_gate, p0, T, hca.ring_k, hca.ring_v, hca.ring_gate)
    return dict(idx=idx, csa_out=out_c, csa_lse=lse_c, hca_out=out_h, hca_lse=lse_h, q_pos=q_pos)
