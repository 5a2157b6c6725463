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

from . import (BF16, E2M1_UE8M0, F32, csa_attend, csa_attend_workspace, csa_cache_append, csa_compress,
               csa_index_key_quantize, csa_index_topk, csa_index_topk_fp4, csa_index_topk_fp4_workspace,
               csa_index_topk_workspace, hca_attend, hca_attend_workspace, hca_cache_append,
               hca_compress, key_storage, swa_ring_write, KV_FP8_K_ROW, KV_FP8_V_ROW)


def _i64(x, device):
    return torch.as_tensor(x, dtype=torch.int64, device=device).reshape(-1).contiguous()


def kv_storage(B, Ncap, d, dtype, kv_fp8, device):
    """Compressed K and V caches: [B, Ncap, d] of dtype, or with kv_fp8 (d = 128, bfloat16 raw
    tokens) the FP8 rows of KV_FP8_K_ROW / KV_FP8_V_ROW bytes (pogovet.com detail 5: KV entries in
    FP8, the RoPE dims in BF16)."""
    if kv_fp8:
        assert d == 128 and dtype == torch.bfloat16
        return (torch.zeros(B, Ncap, KV_FP8_K_ROW, dtype=torch.uint8, device=device),
                torch.zeros(B, Ncap, KV_FP8_V_ROW, dtype=torch.uint8, device=device))
    return (torch.zeros(B, Ncap, d, dtype=dtype, device=device), torch.zeros(B, Ncap, d, dtype=dtype, device=device))


class CSACache:
    """Compressed sparse attention cache of B sequences (m = 4 by default)."""

    def __init__(self, B, Ncap, d, W, d_I, key_fmt, dtype, device="cuda", m=4, kv_fp8=False):
        Ncap = (Ncap + 255) // 256 * 256   # capacity in whole 256-key tensor-core indexer stages
        self.B, self.Ncap, self.d, self.W, self.d_I, self.m = B, Ncap, d, W, d_I, m
        self.key_fmt, self.dtype, self.device, self.kv_fp8 = key_fmt, dtype, device, kv_fp8
        self.ck, self.cv = kv_storage(B, Ncap, d, dtype, kv_fp8, device)
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

    def __init__(self, B, Ncap, d, W, dtype, device="cuda", m=128, kv_fp8=False):
        self.B, self.Ncap, self.d, self.W, self.m, self.dtype, self.device = B, Ncap, d, W, m, dtype, device
        self.kv_fp8 = kv_fp8
        self.ck, self.cv = kv_storage(B, Ncap, d, dtype, kv_fp8, device)
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
        self.ws_topk = torch.zeros(csa_index_topk_workspace(B, 1, cache.Ncap, k), dtype=torch.uint8, device=dev)
        self.ws_att = torch.zeros(max(256, csa_attend_workspace(B, 1, H, d, k, cache.W)), dtype=torch.uint8,
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
        self.ws = torch.zeros(max(256, hca_attend_workspace(B, 1, H, d, cache.Ncap, cache.W, splits)),
                              dtype=torch.uint8, device=dev)

    def step(self, pos, q, k_new, v_new, gate_new):
        c = self.c
        hca_cache_append(k_new, v_new, gate_new, pos, self.slot_bias, c.m, c.ring_k, c.ring_v, c.ring_gate, c.ck,
                         c.cv)
        hca_attend(q, self.scale, c.ck, c.cv, c.m, c.ring_k, c.ring_v, c.W, pos, self.out, self.lse,
                   splits=self.splits, workspace=self.ws)
        return self.out, self.lse


class HybridPrefill:
    """Chunked prefill of chunks of T tokens through a CSA layer and an HCA layer (B sequences, all
    at the same chunk position).  Per chunk: compress its complete blocks into both caches,
    quantise the new index keys, run CSA (indexer, top-k, sparse attention with the causal
    window) and HCA (dense, causal) for every query of the chunk, then move the chunk's last
    tokens into both rings.  Outputs and workspaces are allocated once, so a chunk's calls can be
    captured in a CUDA graph."""

    def __init__(self, csa: CSACache, hca: HCACache, T, H, k, csa_bias, hca_bias, scale=None, H_I=None,
                 q_fp4=False):
        B, d, dev = csa.B, csa.d, csa.device
        # FP4 indexer queries (the keys' MX E2M1 form, quantised per chunk): e2m1 keys only
        self.q_fp4 = q_fp4
        if q_fp4:
            assert csa.key_fmt == E2M1_UE8M0 and H_I is not None
            self.q4c = torch.empty(B, T, H_I, csa.d_I // 2, dtype=torch.uint8, device=dev)
            self.q4s = torch.empty(B, T, H_I, csa.d_I // 32, dtype=torch.uint8, device=dev)
        self.csa, self.hca, self.T, self.H, self.k = csa, hca, T, H, k
        self.csa_bias, self.hca_bias = csa_bias, hca_bias
        self.scale = 1.0 / math.sqrt(d) if scale is None else scale
        self.q_pos = torch.empty(B * T, dtype=torch.int64, device=dev)
        self.p0 = torch.empty(B, dtype=torch.int64, device=dev)
        self.nT = torch.full((B,), T, dtype=torch.int64, device=dev)
        self.idx = torch.empty(B, T, k, dtype=torch.int32, device=dev)
        self.out_c = torch.empty(B, T, H, d, dtype=csa.dtype, device=dev)
        self.lse_c = torch.empty(B, T, H, dtype=torch.float32, device=dev)
        self.out_h = torch.empty(B, T, H, d, dtype=hca.dtype, device=dev)
        self.lse_h = torch.empty(B, T, H, dtype=torch.float32, device=dev)
        ws_topk = (csa_index_topk_fp4_workspace(B, T, H_I, csa.Ncap, k) if q_fp4 else
                   csa_index_topk_workspace(B, T, csa.Ncap, k))
        self.ws_topk = torch.zeros(ws_topk, dtype=torch.uint8, device=dev)
        self.ws_ca = torch.zeros(max(256, csa_attend_workspace(B, T, H, d, k, csa.W)), dtype=torch.uint8, device=dev)
        self.ws_ha = torch.zeros(max(256, hca_attend_workspace(B, T, H, d, hca.Ncap, hca.W, 0)), dtype=torch.uint8,
                                 device=dev)

    def set_position(self, pos0):
        """Position of the next chunk's first token (a multiple of both block sizes)."""
        assert pos0 % self.csa.m == 0 and pos0 % self.hca.m == 0
        B, T, dev = self.csa.B, self.T, self.csa.device
        self.pos0 = int(pos0)
        self.p0.fill_(pos0)
        self.q_pos.copy_((torch.arange(T, device=dev, dtype=torch.int64)[None, :] + pos0).repeat(B, 1).reshape(-1))

    def index_topk(self, q_idx, w, scores_out=None):
        """The chunk's lightning indexer and top-k (bf16 queries, or FP4 queries quantised here)."""
        csa = self.csa
        if self.q_fp4:
            csa_index_key_quantize(q_idx, E2M1_UE8M0, self.q4c, self.q4s)
            csa_index_topk_fp4(self.q4c, self.q4s, w, csa.k_codes, csa.k_scale, self.q_pos, csa.m, self.k, self.idx,
                               scores_out=scores_out, workspace=self.ws_topk)
        else:
            csa_index_topk(q_idx, w, csa.k_codes, csa.k_scale, csa.key_fmt, self.q_pos, csa.m, self.k, self.idx,
                           scores_out=scores_out, workspace=self.ws_topk)

    def step(self, chunk_k, chunk_v, chunk_gate, kidx_chunk, q_csa, q_idx, w, q_hca, scores_out=None):
        """chunk_k/v [B, T, d]; chunk_gate [B, T]; kidx_chunk [B, T // m_csa, d_I] (index keys of the
        new CSA entries); q_csa/q_hca [B, T, H, d]; q_idx [B, T, H_I, d_I]; w [B, T, H_I]."""
        csa, hca, T = self.csa, self.hca, self.T
        csa_compress(chunk_k, chunk_v, chunk_gate, self.p0, self.nT, self.csa_bias, csa.m, csa.ck, csa.cv)
        hca_compress(chunk_k, chunk_v, chunk_gate, self.p0, self.nT, self.hca_bias, hca.m, hca.ck, hca.cv)
        j0, nb = self.pos0 // csa.m, T // csa.m
        for b in range(csa.B):
            csa_index_key_quantize(kidx_chunk[b, :nb], csa.key_fmt, csa.k_codes[b, j0:j0 + nb],
                                   None if csa.k_scale is None else csa.k_scale[b, j0:j0 + nb])
        self.index_topk(q_idx, w, scores_out)
        csa_attend(q_csa, self.scale, csa.ck, csa.cv, self.idx, csa.ring_k, csa.ring_v, csa.W, self.q_pos,
                   self.out_c, self.lse_c, chunk_k=chunk_k, chunk_v=chunk_v, chunk_pos0=self.p0, workspace=self.ws_ca)
        hca_attend(q_hca, self.scale, hca.ck, hca.cv, hca.m, hca.ring_k, hca.ring_v, hca.W, self.q_pos, self.out_h,
                   self.lse_h, chunk_k=chunk_k, chunk_v=chunk_v, chunk_pos0=self.p0, workspace=self.ws_ha)
        swa_ring_write(chunk_k, chunk_v, chunk_gate, self.p0, T, csa.ring_k, csa.ring_v, csa.ring_gate)
        swa_ring_write(chunk_k, chunk_v, chunk_gate, self.p0, T, hca.ring_k, hca.ring_v, hca.ring_gate)
        return dict(idx=self.idx, csa_out=self.out_c, csa_lse=self.lse_c, hca_out=self.out_h, hca_lse=self.lse_h,
                    q_pos=self.q_pos)


def hybrid_prefill_chunk(csa: CSACache, hca: HCACache, pos0, T, chunk_k, chunk_v, chunk_gate, kidx_chunk,
                         q_csa, q_idx, w, q_hca, csa_bias, hca_bias, k, scale=None, scores_out=None):
    """One chunk of T tokens at position pos0 through both layers (see ``HybridPrefill``).
    Returns dict of outputs."""
    step = HybridPrefill(csa, hca, T, q_csa.shape[2], k, csa_bias, hca_bias, scale)
    step.set_position(pos0)
    return step.step(chunk_k, chunk_v, chunk_gate, kidx_chunk, q_csa, q_idx, w, q_hca, scores_out=scores_out)


# ------------------------------------------------------------------ layer-interleave timeline
def interleave_kinds(n_layers: int, mtp: bool = True) -> list[str]:
    """Attention kind of each layer of the stack (pogovet.com article, detail 5): the first two layers
    HCA, then CSA and HCA alternating (CSA first), and an MTP block whose attention is sliding-window
    only ("swa")."""
    kinds = ["hca" if i < 2 else ("csa" if i % 2 == 0 else "hca") for i in range(n_layers)]
    return kinds + (["swa"] if mtp else [])


class SWACache:
    """Sliding-window-only attention state: the ring of the last W raw tokens."""

    def __init__(self, B, d, W, dtype, device="cuda"):
        self.B, self.d, self.W, self.dtype, self.device = B, d, W, dtype, device
        self.ring_k = torch.zeros(B, W, d, dtype=dtype, device=device)
        self.ring_v = torch.zeros(B, W, d, dtype=dtype, device=device)
        self.ring_gate = torch.zeros(B, W, dtype=torch.float32, device=device)
        # attention reads no compressed entry: a one-row placeholder cache and an empty index list
        self.ck = torch.zeros(B, 1, d, dtype=dtype, device=device)
        self.cv = torch.zeros(B, 1, d, dtype=dtype, device=device)

    def build_seq(self, b, k_raw, v_raw, gate, n_ctx):
        _fill_ring(self, b, k_raw, v_raw, gate, n_ctx)


class SWADecode:
    """One decode step of a sliding-window-only layer: the new token into the ring, attention over the
    W most recent tokens (CSA attention with no selected entry)."""

    def __init__(self, cache: SWACache, H, scale=None):
        self.c, self.H = cache, H
        B, d, dev = cache.B, cache.d, cache.device
        self.scale = 1.0 / math.sqrt(d) if scale is None else scale
        self.idx = torch.empty(B, 1, 0, dtype=torch.int32, device=dev)
        self.out = torch.empty(B, 1, H, d, dtype=cache.dtype, device=dev)
        self.lse = torch.empty(B, 1, H, dtype=torch.float32, device=dev)
        self.ws = torch.zeros(max(256, csa_attend_workspace(B, 1, H, d, 0, cache.W)), dtype=torch.uint8, device=dev)

    def step(self, pos, q, k_new, v_new, gate_new):
        c = self.c
        swa_ring_write(k_new, v_new, gate_new, pos, 1, c.ring_k, c.ring_v, c.ring_gate)
        csa_attend(q, self.scale, c.ck, c.cv, self.idx, c.ring_k, c.ring_v, c.W, pos, self.out, self.lse,
                   workspace=self.ws)
        return self.out, self.lse


class InterleavedDecode:
    """One decode step through a stack of attention layers of the kinds given (``interleave_kinds``),
    each with its own cache: CSA layers append, index, select and attend; HCA layers append and attend
    densely; the MTP layer attends over its window.  Per layer the step takes that layer's new token
    (k, v, gate; for CSA also the index-key input), its queries (for CSA also the indexer queries and
    head weights); the calls of all layers can be captured in one CUDA graph.  The layers' inputs are
    independent here (no projections between layers): the timeline is the attention path of the stack."""

    def __init__(self, kinds, caches, H, H_I, k, biases, scale=None):
        assert len(kinds) == len(caches) == len(biases)
        self.kinds, self.caches = list(kinds), list(caches)
        self.steps = []
        for kind, c, bias in zip(kinds, caches, biases):
            if kind == "csa":
                self.steps.append(CSADecode(c, H, H_I, k, bias, scale))
            elif kind == "hca":
                self.steps.append(HCADecode(c, H, bias, scale))
            else:
                self.steps.append(SWADecode(c, H, scale))

    def step(self, pos, inputs):
        """inputs[i]: dict of layer i's tensors -- q, k_new, v_new, gate_new, and for CSA layers
        q_idx, w, kidx_new.  Returns the layers' (out, lse)."""
        outs = []
        for kind, st, x in zip(self.kinds, self.steps, inputs):
            if kind == "csa":
                o, l, _ = st.step(pos, x["q"], x["q_idx"], x["w"], x["k_new"], x["v_new"], x["gate_new"],
                                  x["kidx_new"])
            else:
                o, l = st.step(pos, x["q"], x["k_new"], x["v_new"], x["gate_new"])
            outs.append((o, l))
        return outs
