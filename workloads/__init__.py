"""Seeded synthetic inputs for the CSA + HCA hot path.

This module holds the workload definitions (sizes, dtypes, value distributions) and
the seeded generators that produce their inputs.  It contains none of the method's
arithmetic: no pooling, scoring, selection, quantisation or attention.  Both the CUDA
library's tests/benchmark and the CPU oracle consume what it produces.

Generators are torch generators (CPU, or CUDA for the large workloads); every tensor
is seeded from (workload seed, tensor name, sequence index), so a single sequence of a
large workload can be regenerated on its own.  Values are rounded once to the storage
dtype (bf16 or fp32) by torch.
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch


# --------------------------------------------------------------------------- configs
@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "csa_decode" | "hca_decode" | "hybrid_decode" | "hybrid_prefill" | "pool"
    B: int
    d: int
    H: int
    W: int = 128              # sliding window (= ring capacity)
    m_csa: int = 4
    m_hca: int = 128
    H_I: int = 16
    d_I: int = 64
    k: int = 512
    kv: str = "bf16"          # raw / compressed KV storage dtype: "bf16" | "f32"
    key_fmt: str = "e4m3"     # index-key storage: "f32" | "bf16" | "e4m3" | "e2m1"
    L: tuple = ()             # decode: context length per sequence (incl. the new token)
    L_range: tuple = ()       # decode: lengths drawn uniformly from [lo, hi] (inclusive)
    T: int = 0                # prefill: chunk length
    offset: int = 0           # prefill: position of the chunk's first token
    # value distributions: standard deviations (N(0, std^2)); None -> 1/sqrt(last dim)
    q_std: float | None = 1.0
    kv_std: float | None = 1.0
    qi_std: float | None = 1.0
    ki_std: float | None = 1.0
    gate_std: float = 1.0
    bias_std: float = 0.5
    outlier_frac: float = 0.0
    outlier_mult: float = 4.0
    index_q: str = "bf16"     # indexer queries: "bf16", or "e2m1" (FP4, the keys' MX form)
    kv_cache: str = "bf16"    # compressed K/V storage: "bf16" (= kv), or "fp8" (E4M3, RoPE dims of K in bf16)
    seed: int = 0

    def lengths(self) -> list[int]:
        if self.L:
            return list(self.L)
        lo, hi = self.L_range
        g = torch.Generator().manual_seed(_seed(self.seed, "lengths", 0))
        return [int(x) for x in torch.randint(lo, hi + 1, (self.B,), generator=g)]

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


WORKLOADS = {
    # One sequence, fp32, tiny: L=4096, d=64, 8 heads, indexer 4 x 32, k=64, W=128.
    "tiny_csa_decode_f32": Workload(
        name="tiny_csa_decode_f32", kind="csa_decode", B=1, L=(4096,), d=64, H=8, H_I=4, d_I=32,
        k=64, W=128, kv="f32", key_fmt="f32", q_std=1.0 / 8.0, kv_std=1.0, qi_std=None, ki_std=1.0),
    # Batch 8 x 128K, 64 heads over one KV stream (d=128), fp8 e4m3 index keys, k=512.
    "csa_decode_b8_128k_bf16": Workload(
        name="csa_decode_b8_128k_bf16", kind="csa_decode", B=8, L=(131072,) * 8, d=128, H=64,
        H_I=16, d_I=64, k=512, W=128, kv="bf16", key_fmt="e4m3",
        q_std=None, kv_std=None, qi_std=None, ki_std=None),
    # Batch 4 x 1M, HCA m=128 -> 8192 entries + window 128, 64 heads, d=128.
    "hca_decode_b4_1m_bf16": Workload(
        name="hca_decode_b4_1m_bf16", kind="hca_decode", B=4, L=(1 << 20,) * 4, d=128, H=64,
        W=128, kv="bf16", q_std=None, kv_std=1.0),
    # One chunk of 4096 queries at offset 262144, CSA k=1024 + HCA dense, bf16 index keys.
    "hybrid_prefill_t4096_at_256k_bf16": Workload(
        name="hybrid_prefill_t4096_at_256k_bf16", kind="hybrid_prefill", B=1, T=4096, offset=262144,
        d=128, H=64, H_I=16, d_I=64, k=1024, W=128, kv="bf16", key_fmt="bf16"),
    # Batch 32, lengths U[512K, 1M]; a CSA layer (k=1024, e2m1 index keys) then an HCA layer.
    "decode_1m_b32_csa_hca": Workload(
        name="decode_1m_b32_csa_hca", kind="hybrid_decode", B=32, L_range=(524288, 1048576),
        d=128, H=64, H_I=16, d_I=64, k=1024, W=128, kv="bf16", key_fmt="e2m1",
        outlier_frac=0.01),
}

# Bulk pooling of one 1M-token sequence into both compressed caches (CSA m=4, HCA m=128), bf16, d=128.
WORKLOADS["pool_1m_bf16"] = Workload(name="pool_1m_bf16", kind="pool", B=1, L=(1 << 20,), d=128, H=64, kv="bf16",
                                     kv_std=1.0)

# The 1M-context decode workload with the lightning indexer's queries in FP4 as well.
WORKLOADS["decode_1m_b32_csa_hca_q4"] = replace(WORKLOADS["decode_1m_b32_csa_hca"], name="decode_1m_b32_csa_hca_q4",
                                               index_q="e2m1")

KEY_FMT_CODE = {"f32": 0, "bf16": 1, "e4m3": 2, "e2m1": 3}


def shrink(w: Workload, **kw) -> Workload:
    """A smaller variant of a workload (same distributions), for fast tests."""
    return replace(w, **kw)


# ------------------------------------------------------------------------ generators
def _seed(base: int, name: str, b: int) -> int:
    h = hashlib.sha256(f"{base}/{name}/{b}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, base: int, name: str, b: int) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev) if dev.type == "cuda" else torch.Generator()
    g.manual_seed(_seed(base, name, b))
    return g


def torch_dtype(kind: str):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[kind]


def normal(shape, std, device, base, name, b, dtype=torch.float32):
    g = _gen(device, base, name, b)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def uniform(shape, device, base, name, b):
    g = _gen(device, base, name, b)
    return torch.rand(*shape, generator=g, device=device, dtype=torch.float32)


def _std(v, dim):
    return (1.0 / math.sqrt(dim)) if v is None else float(v)


def outlier_rows(n: int, frac: float, device, base: int, name: str, b: int):
    """Seeded choice of round(frac*n) row indices (the rows to be given outlier magnitude)."""
    cnt = int(round(frac * n))
    if cnt == 0:
        return torch.zeros(0, dtype=torch.long, device=device)
    g = _gen(device, base, name, b)
    return torch.randperm(n, generator=g, device=device)[:cnt]


def layer_bias(w: Workload, layer: str, m: int, device="cpu"):
    """Learned per-slot position bias of a layer's compressor, [m] fp32."""
    return normal((m,), w.bias_std, device, w.seed, f"{layer}/bias", 0)


def raw_tokens(w: Workload, layer: str, b: int, n: int, device="cpu", pos0: int = 0, tag="raw"):
    """Raw K, V [n, d] (storage dtype) and gate logits [n] fp32 of sequence b.

    ``pos0`` only names the stream: tokens of a sequence are generated as one stream
    starting at ``pos0`` (prefill chunks use their own stream)."""
    dt = torch_dtype(w.kv)
    std = _std(w.kv_std, w.d)
    name = f"{layer}/{tag}@{pos0}"
    k = normal((n, w.d), std, device, w.seed, name + "/k", b)
    v = normal((n, w.d), std, device, w.seed, name + "/v", b)
    if w.outlier_frac > 0:
        rows = outlier_rows(n, w.outlier_frac, device, w.seed, name + "/outliers", b)
        k[rows] *= w.outlier_mult
        v[rows] *= w.outlier_mult
    gate = normal((n,), w.gate_std, device, w.seed, name + "/gate", b)
    return k.to(dt), v.to(dt), gate


def index_key_inputs(w: Workload, layer: str, b: int, n: int, device="cpu", tag="kidx"):
    """Index-key inputs, one row per compressed CSA entry, [n, d_I] (bf16, or fp32 when the
    key format is fp32)."""
    dt = torch.float32 if w.key_fmt == "f32" else torch.bfloat16
    x = normal((n, w.d_I), _std(w.ki_std, w.d_I), device, w.seed, f"{layer}/{tag}", b)
    if w.outlier_frac > 0:
        rows = outlier_rows(n, w.outlier_frac, device, w.seed, f"{layer}/{tag}/outliers", b)
        x[rows] *= w.outlier_mult
    return x.to(dt)


def queries(w: Workload, layer: str, b: int, T: int = 1, device="cpu", tag="q"):
    """Attention queries [T, H, d] (storage dtype)."""
    return normal((T, w.H, w.d), _std(w.q_std, w.d), device, w.seed, f"{layer}/{tag}", b).to(torch_dtype(w.kv))


def indexer_queries(w: Workload, layer: str, b: int, T: int = 1, device="cpu", tag="qi"):
    """Indexer queries [T, H_I, d_I] and head weights w [T, H_I] ~ U(0,1)."""
    dt = torch.float32 if w.key_fmt == "f32" else torch.bfloat16
    qi = normal((T, w.H_I, w.d_I), _std(w.qi_std, w.d_I), device, w.seed, f"{layer}/{tag}", b).to(dt)
    wt = uniform((T, w.H_I), device, w.seed, f"{layer}/{tag}/w", b)
    return qi, wt


# --------------------------------------------------------------------- host helpers
def to_numpy(t: torch.Tensor) -> np.ndarray:
    """Host copy for the oracle: fp32 as float32, bf16 as its uint16 bit pattern."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    return t.numpy()


def prefill_inputs(w: Workload, device="cuda", b: int = 0):
    """Inputs of one chunked-prefill problem for sequence b (synthetic prior state + chunk).

    Prior state before the chunk (all values drawn, not computed): offset/m_csa CSA entries and
    their index-key inputs, offset/m_hca HCA entries, and the W raw tokens before the chunk (the
    window ring).  The chunk: T raw tokens (K, V, gate), T/m_csa index-key inputs for the CSA
    entries it completes, and per query: CSA and HCA queries, indexer queries and head weights.
    """
    dt = torch_dtype(w.kv)
    kdt = torch.float32 if w.key_fmt == "f32" else torch.bfloat16
    n_csa, n_hca = w.offset // w.m_csa, w.offset // w.m_hca
    std = _std(w.kv_std, w.d)
    out = dict(
        csa_ck=normal((n_csa, w.d), std, device, w.seed, "prior/csa/ck", b, dt),
        csa_cv=normal((n_csa, w.d), std, device, w.seed, "prior/csa/cv", b, dt),
        csa_kidx=normal((n_csa, w.d_I), _std(w.ki_std, w.d_I), device, w.seed, "prior/csa/kidx", b, kdt),
        hca_ck=normal((n_hca, w.d), std, device, w.seed, "prior/hca/ck", b, dt),
        hca_cv=normal((n_hca, w.d), std, device, w.seed, "prior/hca/cv", b, dt),
        csa_bias=layer_bias(w, "csa", w.m_csa, device),
        hca_bias=layer_bias(w, "hca", w.m_hca, device),
    )
    out["ring_k"], out["ring_v"], out["ring_gate"] = raw_tokens(w, "prior", b, w.W, device, tag="ring")
    out["chunk_k"], out["chunk_v"], out["chunk_gate"] = raw_tokens(w, "chunk", b, w.T, device, pos0=w.offset)
    out["chunk_kidx"] = index_key_inputs(w, "chunk", b, w.T // w.m_csa, device)
    out["q_csa"] = queries(w, "csa", b, w.T, device)
    out["q_hca"] = queries(w, "hca", b, w.T, device)
    out["q_idx"], out["w"] = indexer_queries(w, "csa", b, w.T, device)
    return out

# The 1M-context decode workload with the compressed K/V caches in FP8 (the RoPE dims of K in BF16).
WORKLOADS["decode_1m_b32_csa_hca_kv8"] = replace(WORKLOADS["decode_1m_b32_csa_hca"], name="decode_1m_b32_csa_hca_kv8",
                                                kv_cache="fp8")

# The prefill chunk with the lightning indexer in FP4 for both operands (e2m1 keys, FP4 queries).
WORKLOADS["hybrid_prefill_t4096_at_256k_q4"] = replace(WORKLOADS["hybrid_prefill_t4096_at_256k_bf16"],
                                                      name="hybrid_prefill_t4096_at_256k_q4", key_fmt="e2m1",
                                                      index_q="e2m1")
