"""CPU oracle for CSA + HCA hybrid compressed attention -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct restatement of the method in fp64 (scalar C in
``oracle.c`` plus thin numpy glue here).  It is used by the tests, by
``__graft_entry__.smoke()`` and by the benchmark's CPU-baseline leg, and by
nothing else: the product path never imports it.  It shares no code with the
CUDA library.

Sources (titles of the pages the method is described on):
  * honbul.tistory.com/221 -- sections "CSA: 압축한 뒤, 필요한 기억만 골라서 보기",
    "HCA: 더 강하게 압축하고, 압축된 전체를 보기", "KV cache를 줄이는 방식".
  * pogovet.com, "DeepSeek-V4: a million-token context that agents can actually
    use" -- detail 4 "CSA와 HCA를 결합한 하이브리드 어텐션" (m=4 softmax-gated
    pooling with a learned position bias, lightning indexer with top-k, sliding
    window; HCA with m=128 and dense attention), detail 5 (FP4 indexer).

Array conventions: float arrays are ``np.float32``; bfloat16 arrays are passed as
their raw bits in ``np.uint16``.  Every function returns fp64 results unless it
says otherwise.

Parity pins: every function here is pinned by tests in ``tests/test_oracle_*.py``
(closed forms, special cases that reduce to textbook routines, brute force on tiny
inputs, exhaustive code tables).  No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 2              # storage dtype codes (F64: dequantised values passed back in)
KEY_F32, KEY_BF16, KEY_E4M3, KEY_E2M1 = 0, 1, 2, 3   # index-key formats


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            D = ctypes.c_double
            lib.oc_double_to_bf16.argtypes = [D]
            lib.oc_double_to_bf16.restype = ctypes.c_uint16
            lib.oc_round_bf16.argtypes = [P, I64, P]
            lib.oc_pool.argtypes = [P, I, P, P, I, I64, I, P, P]
            lib.oc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oc_e4m3_decode.restype = D
            lib.oc_e4m3_encode.argtypes = [D]
            lib.oc_e4m3_encode.restype = ctypes.c_uint8
            lib.oc_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.oc_e2m1_decode.restype = D
            lib.oc_e2m1_encode.argtypes = [D]
            lib.oc_e2m1_encode.restype = ctypes.c_uint8
            lib.oc_quant_e4m3_rowscale.argtypes = [P, I, I64, I, P, P]
            lib.oc_quant_e2m1_ue8m0.argtypes = [P, I, I64, I, P, P]
            lib.oc_dequant_keys.argtypes = [I, P, P, I64, I, P]
            lib.oc_quant_kv_fp8.argtypes = [P, I64, I, I, P, P, P]
            lib.oc_dequant_kv_fp8.argtypes = [P, P, P, I64, I, I, P]
            lib.oc_index_scores.argtypes = [P, I, P, I, I, I, P, I64, P, P]
            lib.oc_topk.argtypes = [P, I64, I, P, I, P]
            lib.oc_attend.argtypes = [P, I, I, I, D, P, P, I, P, I64, P, P, I, P, I64, P, P]
            lib.oc_lse_merge.argtypes = [P, P, I, I, I, P, P]
            lib.oc_num_threads.restype = I
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _dt(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"oracle storage arrays are float32, float64 or uint16 (bf16 bits), got {a.dtype}")


def num_threads() -> int:
    return int(_L().oc_num_threads())


# ------------------------------------------------------------------ conversions
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(a: np.ndarray) -> np.ndarray:
    return bf16_to_f64(a) if a.dtype == np.uint16 else np.asarray(a, dtype=np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _L().oc_round_bf16(_p(x), x.size, _p(out))
    return out


def round_to(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round once to the storage dtype (F32 -> float32, BF16 -> uint16 bits)."""
    return round_bf16(x) if dtype == BF16 else np.ascontiguousarray(x, dtype=np.float64).astype(np.float32)


# ------------------------------------------------------------- a1/a2: pooling
def pool(x: np.ndarray, gate: np.ndarray, bias: np.ndarray, m: int, n_blocks: int | None = None):
    """Softmax-gated pooling of blocks of m tokens (one gate per token, bias per slot).

    x: [>= n_blocks*m, d]; gate: [>= n_blocks*m] float32; bias: [m] float32.
    Returns (pooled [n_blocks, d] fp64, alpha [n_blocks, m] fp64).
    """
    x = np.ascontiguousarray(x)
    d = x.shape[-1]
    if n_blocks is None:
        n_blocks = x.shape[0] // m
    gate = np.ascontiguousarray(gate, dtype=np.float32)
    bias = np.ascontiguousarray(bias, dtype=np.float32)
    assert bias.shape == (m,) and gate.shape[0] >= n_blocks * m and x.shape[0] >= n_blocks * m
    out = np.empty((n_blocks, d), dtype=np.float64)
    alpha = np.empty((n_blocks, m), dtype=np.float64)
    _L().oc_pool(_p(x), _dt(x), _p(gate), _p(bias), m, n_blocks, d, _p(out), _p(alpha))
    return out, alpha


# -------------------------------------------------------- a4: key quantisation
def e4m3_decode(code: int) -> float:
    return float(_L().oc_e4m3_decode(code))


def e4m3_encode(y: float) -> int:
    return int(_L().oc_e4m3_encode(float(y)))


def e2m1_decode(code: int) -> float:
    return float(_L().oc_e2m1_decode(code))


def e2m1_encode(y: float) -> int:
    return int(_L().oc_e2m1_encode(float(y)))


def quant_e4m3_rowscale(x: np.ndarray):
    """Returns (codes uint8 [rows, d], scale float32 [rows])."""
    x = np.ascontiguousarray(x)
    rows, d = x.shape
    codes = np.empty((rows, d), dtype=np.uint8)
    scale = np.empty((rows,), dtype=np.float32)
    _L().oc_quant_e4m3_rowscale(_p(x), _dt(x), rows, d, _p(codes), _p(scale))
    return codes, scale


def quant_e2m1_ue8m0(x: np.ndarray):
    """Returns (packed uint8 [rows, d/2], biased exponents uint8 [rows, d/32])."""
    x = np.ascontiguousarray(x)
    rows, d = x.shape
    assert d % 32 == 0
    packed = np.empty((rows, d // 2), dtype=np.uint8)
    se = np.empty((rows, d // 32), dtype=np.uint8)
    _L().oc_quant_e2m1_ue8m0(_p(x), _dt(x), rows, d, _p(packed), _p(se))
    return packed, se


def quantize_keys(x: np.ndarray, fmt: int):
    """Index keys in storage format ``fmt``: returns (codes, scales-or-None)."""
    if fmt == KEY_F32:
        return np.ascontiguousarray(x, dtype=np.float32), None
    if fmt == KEY_BF16:
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x), None
    if fmt == KEY_E4M3:
        return quant_e4m3_rowscale(x)
    if fmt == KEY_E2M1:
        return quant_e2m1_ue8m0(x)
    raise ValueError(fmt)


def dequant_keys(fmt: int, codes: np.ndarray, scales, d: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes)
    rows = codes.shape[0]
    out = np.empty((rows, d), dtype=np.float64)
    sp = _p(np.ascontiguousarray(scales)) if scales is not None else None
    _L().oc_dequant_keys(fmt, _p(codes), sp, rows, d, _p(out))
    return out


def quant_kv_fp8(x: np.ndarray, d_keep: int):
    """FP8 storage of compressed K/V rows (see ``oc_quant_kv_fp8``): x [rows, d] (any float dtype,
    taken as fp64).  Returns (codes uint8 [rows, d - d_keep], scales uint8 [rows, (d - d_keep)/64],
    keep uint16 BF16 bits [rows, d_keep])."""
    x = np.ascontiguousarray(to_f64(x) if x.dtype == np.uint16 else x, dtype=np.float64)
    rows, d = x.shape
    assert (d - d_keep) % 64 == 0 and 0 <= d_keep <= d
    codes = np.empty((rows, d - d_keep), dtype=np.uint8)
    scales = np.empty((rows, (d - d_keep) // 64), dtype=np.uint8)
    keep = np.zeros((rows, max(d_keep, 1)), dtype=np.uint16)
    _L().oc_quant_kv_fp8(_p(x), rows, d, d_keep, _p(codes), _p(scales), _p(keep))
    return codes, scales, keep[:, :d_keep]


def dequant_kv_fp8(codes: np.ndarray, scales: np.ndarray, keep: np.ndarray, d: int) -> np.ndarray:
    codes, scales = np.ascontiguousarray(codes), np.ascontiguousarray(scales)
    rows = codes.shape[0]
    d_keep = d - codes.shape[1]
    kp = np.ascontiguousarray(keep if d_keep else np.zeros((rows, 1), dtype=np.uint16))
    out = np.empty((rows, d), dtype=np.float64)
    _L().oc_dequant_kv_fp8(_p(codes), _p(scales), _p(kp), rows, d, d_keep, _p(out))
    return out


def fp4_query(q_idx: np.ndarray) -> np.ndarray:
    """Indexer queries in FP4, as the lightning indexer's query-key path runs it (honbul.tistory
    .com/221, section on FP4 QAT of the CSA indexer's query-key path; pogovet.com detail 5, the
    indexer runs in FP4): every run of 32 consecutive elements of a head's vector is quantised
    with the same MX rule as the index keys -- e = the smallest integer with amax <= 6 * 2^e
    (0 for an all-zero run), code = RNE_e2m1(x * 2^-e) -- and the query becomes 2^e * code.

    q_idx: [T, H_I, d_I] (float32 or bf16 bits), d_I % 32 == 0.  Returns fp64 [T, H_I, d_I]."""
    q_idx = np.ascontiguousarray(q_idx)
    T, H_I, d_I = q_idx.shape
    codes, se = quant_e2m1_ue8m0(q_idx.reshape(T * H_I, d_I))
    return dequant_keys(KEY_E2M1, codes, se, d_I).reshape(T, H_I, d_I)


# ------------------------------------------------------------ a5: indexer
def index_scores(q_idx: np.ndarray, w: np.ndarray, khat: np.ndarray, n_vis) -> np.ndarray:
    """I(t,s) = sum_h w[t,h] * relu(q[t,h,:] . khat[s,:]); -inf for s >= n_vis[t].

    q_idx: [T, H_I, d_I]; w: [T, H_I] float32; khat: [N, d_I] fp64.  Returns [T, N] fp64.
    """
    q_idx = np.ascontiguousarray(q_idx)
    T, H_I, d_I = q_idx.shape
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(T, H_I)
    khat = np.ascontiguousarray(khat, dtype=np.float64)
    N = khat.shape[0]
    nv = np.ascontiguousarray(np.broadcast_to(np.asarray(n_vis, dtype=np.int64), (T,)))
    S = np.empty((T, N), dtype=np.float64)
    _L().oc_index_scores(_p(q_idx), _dt(q_idx), _p(w), T, H_I, d_I, _p(khat), N, _p(nv), _p(S))
    return S


# ---------------------------------------------------------------- a6: top-k
def topk(S: np.ndarray, n_vis, k: int) -> np.ndarray:
    """Top-k per row (score desc, ties -> lower index), ascending index order, -1 padded."""
    S = np.ascontiguousarray(np.atleast_2d(S), dtype=np.float64)
    R, N = S.shape
    nv = np.ascontiguousarray(np.broadcast_to(np.asarray(n_vis, dtype=np.int64), (R,)))
    assert (nv <= N).all()
    idx = np.empty((R, k), dtype=np.int32)
    _L().oc_topk(_p(S), N, R, _p(nv), k, _p(idx))
    return idx


# -------------------------------------------------------- a7/a8: attention
def attend(q: np.ndarray, scale: float, kc, vc, c_rows, kw, vw, w_rows):
    """Joint softmax attention of all heads of one query over compressed rows
    ``kc/vc[c_rows]`` together with raw window rows ``kw/vw[w_rows]``.

    q: [H, d].  Returns (o [H, d] fp64, lse [H] fp64).
    """
    q = np.ascontiguousarray(q)
    H, d = q.shape
    c_rows = np.ascontiguousarray(np.asarray(c_rows, dtype=np.int64).ravel())
    w_rows = np.ascontiguousarray(np.asarray(w_rows, dtype=np.int64).ravel())
    if kc is None:
        kc = vc = np.zeros((1, d), dtype=np.float32)
        assert c_rows.size == 0
    if kw is None:
        kw = vw = np.zeros((1, d), dtype=np.float32)
        assert w_rows.size == 0
    kc, vc, kw, vw = (np.ascontiguousarray(a) for a in (kc, vc, kw, vw))
    assert _dt(kc) == _dt(vc) and _dt(kw) == _dt(vw)
    assert c_rows.size == 0 or (c_rows.min() >= 0 and c_rows.max() < kc.shape[0])
    assert w_rows.size == 0 or (w_rows.min() >= 0 and w_rows.max() < kw.shape[0])
    o = np.empty((H, d), dtype=np.float64)
    lse = np.empty((H,), dtype=np.float64)
    _L().oc_attend(_p(q), _dt(q), H, d, float(scale),
                   _p(kc), _p(vc), _dt(kc), _p(c_rows), c_rows.size,
                   _p(kw), _p(vw), _dt(kw), _p(w_rows), w_rows.size, _p(o), _p(lse))
    return o, lse


def lse_merge(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Exact merge of S partial softmax results: o_parts [S,H,d], lse_parts [S,H]."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    S, H, d = o_parts.shape
    o = np.empty((H, d), dtype=np.float64)
    lse = np.empty((H,), dtype=np.float64)
    _L().oc_lse_merge(_p(o_parts), _p(lse_parts), S, H, d, _p(o), _p(lse))
    return o, lse


from .reference import *  # noqa: E402,F401,F403  (step-by-step compositions)
