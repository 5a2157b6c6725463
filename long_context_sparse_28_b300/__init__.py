"""Thin Python binding of ``libcsahca.so`` -- CSA + HCA hybrid compressed attention on B300.

Every function here has the name of the C entry point it calls (see ``include/csa_hca.h``)
and only marshals arguments: it reads sizes off torch tensors, passes raw device pointers
and the current CUDA stream, and raises ``CsaHcaError`` on a non-OK status.  All arithmetic
runs in the library's CUDA kernels.  The library must have been built
(``python -m long_context_sparse_28_b300.build_lib``); importing this module without it
raises immediately -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsahca.so")

F32, BF16, E4M3_ROWSCALE, E2M1_UE8M0 = 0, 1, 2, 3
KEY_FMT = {"f32": F32, "bf16": BF16, "e4m3": E4M3_ROWSCALE, "e2m1": E2M1_UE8M0}
# compressed K/V in FP8 with the RoPE dims of K in bf16: caches are uint8 tensors of these row sizes
KV_FP8, KV_FP8_K_ROW, KV_FP8_V_ROW = 4, 224, 128

# every C entry point and its ctypes signature
_P, _I64, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "csa_compress": ([_P, _P, _P, _I64, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I64, _P], _I),
    "hca_compress": ([_P, _P, _P, _I64, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I64, _P], _I),
    "csa_index_key_quantize": ([_P, _I, _I64, _I, _I, _P, _P, _P], _I),
    "csa_index_topk": ([_P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I64, _I, _I, _P, _P, _P, _SZ, _P], _I),
    "csa_index_topk_workspace": ([_I, _I, _I64, _I], _SZ),
    "csa_index_topk_fp4_workspace": ([_I, _I, _I, _I64, _I], _SZ),
    "csa_index_topk_fp4": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _I64, _I, _I, _P, _P, _P, _SZ, _P], _I),
    "csa_index_scores": ([_P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I64, _I, _P, _P], _I),
    "csa_topk_from_scores": ([_P, _I64, _I, _P, _I, _P, _P, _SZ, _P], _I),
    "csa_topk_workspace": ([_I, _I64, _I], _SZ),
    "csa_attend": ([_P, _I, _I, _I, _I, _F, _P, _P, _I64, _P, _I, _P, _P, _I, _I, _P, _P, _P, _I64, _P, _I, _P,
                    _P, _P, _SZ, _P], _I),
    "csa_attend_workspace": ([_I, _I, _I, _I, _I, _I], _SZ),
    "hca_attend": ([_P, _I, _I, _I, _I, _F, _P, _P, _I64, _I, _P, _P, _I, _I, _P, _P, _P, _I64, _P, _I, _I, _P,
                    _P, _P, _SZ, _P], _I),
    "hca_attend_workspace": ([_I, _I, _I, _I, _I64, _I, _I], _SZ),
    "hca_attend_noalloc": ([_P, _I, _I, _I, _I, _F, _P, _P, _I64, _I, _P, _P, _I, _I, _P, _P, _P, _I64, _P, _I, _I,
                            _P, _P, _P], _I),
    "hca_attend_noalloc_scratch_bytes": ([], _SZ),
    "csa_cache_append": ([_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _I, _P, _P, _P, _I, _P, _P, _I64, _P, _P,
                          _I, _I, _P], _I),
    "hca_cache_append": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _P, _P, _I, _P, _P, _I64, _P], _I),
    "swa_ring_write": ([_P, _P, _P, _I64, _P, _I, _I, _I, _I, _P, _P, _P, _I, _P], _I),
    "csahca_device_status": ([_P], _I),
    "csahca_status_string": ([_I], ctypes.c_char_p),
    "csahca_launch_count": ([], ctypes.c_uint64),
    "csahca_selftest_bounded_wait": ([ctypes.c_uint64, _P], _I),
    "csahca_version": ([], _I),
}


class CsaHcaError(RuntimeError):
    pass


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"CUDA library not built: {LIB_PATH} is missing "
                          "(run python -m long_context_sparse_28_b300.build_lib)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = None


def library():
    """The loaded ``libcsahca.so`` (loaded on first use; raises ImportError if it is not built)."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


# ----------------------------------------------------------------------------- helpers
def _p(t):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "tensors passed to the library must be contiguous CUDA tensors"
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dt(t) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _kv_dt(x, ck) -> int:
    """kv_dtype of a pooling / append / attention call: FP8 caches (uint8 rows), else x's dtype."""
    return KV_FP8 if ck.dtype == torch.uint8 else _dt(x)


def _check(st: int, name: str):
    if st != 0:
        raise CsaHcaError(f"{name}: {library().csahca_status_string(st).decode()} (status {st})")


def _ws(nbytes: int, device, workspace):
    if workspace is not None:
        assert workspace.numel() * workspace.element_size() >= nbytes
        return workspace, workspace.numel() * workspace.element_size()
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device), max(int(nbytes), 256)


def status_string(st: int) -> str:
    return library().csahca_status_string(st).decode()


def device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error word's status."""
    return int(library().csahca_device_status(_stream(stream)))


def selftest_bounded_wait(limit_ns: int, stream=None) -> None:
    """Runs the library's bounded-wait self-test (a device wait that nothing completes gives up
    after ``limit_ns``); read the outcome with ``device_status()``."""
    _check(library().csahca_selftest_bounded_wait(int(limit_ns), _stream(stream)), "csahca_selftest_bounded_wait")


def launch_count() -> int:
    return int(library().csahca_launch_count())


def version() -> int:
    return int(library().csahca_version())


def key_storage(B: int, Ncap: int, d_I: int, fmt: int, device="cuda"):
    """Allocates index-key storage of a format: (codes, scales-or-None)."""
    if fmt == F32:
        return torch.empty(B, Ncap, d_I, dtype=torch.float32, device=device), None
    if fmt == BF16:
        return torch.empty(B, Ncap, d_I, dtype=torch.bfloat16, device=device), None
    if fmt == E4M3_ROWSCALE:
        return (torch.empty(B, Ncap, d_I, dtype=torch.uint8, device=device),
                torch.empty(B, Ncap, dtype=torch.float32, device=device))
    return (torch.empty(B, Ncap, d_I // 2, dtype=torch.uint8, device=device),
            torch.empty(B, Ncap, d_I // 32, dtype=torch.uint8, device=device))


# ------------------------------------------------------------------------ entry points
def _compress(name, k_raw, v_raw, gate, raw_pos0, n_raw, slot_bias, m, ck, cv, stream):
    B, stride, d = k_raw.shape
    fn = getattr(library(), name)
    _check(fn(_p(k_raw), _p(v_raw), _p(gate), stride, _p(raw_pos0), _p(n_raw), _p(slot_bias), int(m), B, d,
              _kv_dt(k_raw, ck), _p(ck), _p(cv), ck.shape[1], _stream(stream)), name)


def csa_compress(k_raw, v_raw, gate, raw_pos0, n_raw, slot_bias, m, ck, cv, stream=None):
    """k_raw/v_raw [B, raw_stride, d]; gate [B, raw_stride]; raw_pos0/n_raw int64 [B]; ck/cv [B, Ncap, d]."""
    _compress("csa_compress", k_raw, v_raw, gate, raw_pos0, n_raw, slot_bias, m, ck, cv, stream)


def hca_compress(k_raw, v_raw, gate, raw_pos0, n_raw, slot_bias, m, ck, cv, stream=None):
    _compress("hca_compress", k_raw, v_raw, gate, raw_pos0, n_raw, slot_bias, m, ck, cv, stream)


def csa_index_key_quantize(k_in, key_fmt, k_codes, k_scale=None, stream=None):
    """k_in [rows..., d_I] fp32/bf16 -> k_codes/k_scale in key_fmt (same leading rows)."""
    d_I = k_in.shape[-1]
    rows = k_in.numel() // d_I
    _check(library().csa_index_key_quantize(_p(k_in), _dt(k_in), rows, d_I, int(key_fmt), _p(k_codes), _p(k_scale),
                                       _stream(stream)), "csa_index_key_quantize")


def csa_index_topk_workspace(B, T, Ncap, k) -> int:
    return int(library().csa_index_topk_workspace(B, T, Ncap, k))


def csa_index_topk_fp4_workspace(B, T, H_I, Ncap, k) -> int:
    return int(library().csa_index_topk_fp4_workspace(B, T, H_I, Ncap, k))


def csa_index_topk(q_idx, w, k_codes, k_scale, key_fmt, q_pos, m, k, idx_out, scores_out=None,
                   workspace=None, stream=None):
    """q_idx [B, T, H_I, d_I]; w [B, T, H_I]; k_codes/k_scale index keys [B, Ncap, ...];
    q_pos int64 [B*T]; idx_out int32 [B, T, k]; scores_out optional fp32 [B, T, Ncap]."""
    B, T, H_I, d_I = q_idx.shape
    Ncap = k_codes.shape[1]
    ws, nb = _ws(csa_index_topk_workspace(B, T, Ncap, k), q_idx.device, workspace)
    _check(library().csa_index_topk(_p(q_idx), _dt(q_idx), _p(w), _p(k_codes), _p(k_scale), int(key_fmt), B, T, H_I,
                               d_I, _p(q_pos), Ncap, int(m), int(k), _p(idx_out), _p(scores_out), _p(ws), nb,
                               _stream(stream)), "csa_index_topk")


def csa_index_topk_fp4(q_codes, q_scale, w, k_codes, k_scale, q_pos, m, k, idx_out, scores_out=None, workspace=None,
                       stream=None):
    """q_codes [B, T, H_I, d_I/2] uint8 and q_scale [B, T, H_I, d_I/32] uint8: FP4 (MX E2M1) queries;
    keys in CSAHCA_E2M1_UE8M0 form."""
    B, T, H_I, half = q_codes.shape
    d_I = 2 * half
    Ncap = k_codes.shape[1]
    ws, nb = _ws(csa_index_topk_fp4_workspace(B, T, H_I, Ncap, k), q_codes.device, workspace)
    _check(library().csa_index_topk_fp4(_p(q_codes), _p(q_scale), _p(w), _p(k_codes), _p(k_scale), B, T, H_I, d_I,
                                        _p(q_pos), Ncap, int(m), int(k), _p(idx_out), _p(scores_out), _p(ws), nb,
                                        _stream(stream)), "csa_index_topk_fp4")


def csa_index_scores(q_idx, w, k_codes, k_scale, key_fmt, q_pos, m, scores, stream=None):
    """Indexer scores only: scores fp32 [B, T, Ncap] (visible entries written)."""
    B, T, H_I, d_I = q_idx.shape
    Ncap = k_codes.shape[1]
    assert scores.shape[-1] == Ncap
    _check(library().csa_index_scores(_p(q_idx), _dt(q_idx), _p(w), _p(k_codes), _p(k_scale), int(key_fmt), B, T, H_I,
                                 d_I, _p(q_pos), Ncap, int(m), _p(scores), _stream(stream)), "csa_index_scores")


def csa_topk_workspace(R, row_stride, k) -> int:
    return int(library().csa_topk_workspace(R, row_stride, k))


def csa_topk_from_scores(scores, n_vis, k, idx_out, workspace=None, stream=None):
    """scores fp32 [R, row_stride]; n_vis int64 [R]; idx_out int32 [R, k]."""
    R, stride = scores.shape
    ws, nb = _ws(csa_topk_workspace(R, stride, k), scores.device, workspace)
    _check(library().csa_topk_from_scores(_p(scores), stride, R, _p(n_vis), int(k), _p(idx_out), _p(ws), nb,
                                     _stream(stream)), "csa_topk_from_scores")


def csa_attend_workspace(B, T, H, d, k, W) -> int:
    return int(library().csa_attend_workspace(B, T, H, d, k, W))


def hca_attend_workspace(B, T, H, d, Ncap, W, splits=0) -> int:
    return int(library().hca_attend_workspace(B, T, H, d, Ncap, W, splits))


def _chunk_args(chunk_k, chunk_v, chunk_pos0):
    if chunk_k is None:
        return None, None, None, 0
    return chunk_k, chunk_v, chunk_pos0, chunk_k.shape[1]


def csa_attend(q, scale, ck, cv, idx, ring_k, ring_v, W, q_pos, out, lse=None, chunk_k=None, chunk_v=None,
               chunk_pos0=None, workspace=None, stream=None):
    """q/out [B, T, H, d]; ck/cv [B, Ncap, d]; idx int32 [B, T, k]; ring_k/ring_v [B, ring_cap, d];
    q_pos int64 [B*T]; lse optional fp32 [B, T, H]; chunk_* for chunked prefill."""
    B, T, H, d = q.shape
    k = idx.shape[-1]
    ring_cap = ring_k.shape[1] if ring_k is not None else 0
    ck_, cv_, cp_, cs_ = _chunk_args(chunk_k, chunk_v, chunk_pos0)
    ws, nb = _ws(csa_attend_workspace(B, T, H, d, k, W), q.device, workspace)
    _check(library().csa_attend(_p(q), B, T, H, d, float(scale), _p(ck), _p(cv), ck.shape[1], _p(idx), k, _p(ring_k),
                           _p(ring_v), ring_cap, int(W), _p(ck_), _p(cv_), _p(cp_), cs_, _p(q_pos), _kv_dt(q, ck), _p(out),
                           _p(lse), _p(ws), nb, _stream(stream)), "csa_attend")


def hca_attend(q, scale, ck, cv, m, ring_k, ring_v, W, q_pos, out, lse=None, chunk_k=None, chunk_v=None,
               chunk_pos0=None, splits=0, workspace=None, stream=None):
    """Dense HCA attention; arguments as csa_attend, m = HCA block size."""
    B, T, H, d = q.shape
    ring_cap = ring_k.shape[1] if ring_k is not None else 0
    ck_, cv_, cp_, cs_ = _chunk_args(chunk_k, chunk_v, chunk_pos0)
    ws, nb = _ws(hca_attend_workspace(B, T, H, d, ck.shape[1], W, splits), q.device, workspace)
    _check(library().hca_attend(_p(q), B, T, H, d, float(scale), _p(ck), _p(cv), ck.shape[1], int(m), _p(ring_k),
                           _p(ring_v), ring_cap, int(W), _p(ck_), _p(cv_), _p(cp_), cs_, _p(q_pos), int(splits),
                           _kv_dt(q, ck), _p(out), _p(lse), _p(ws), nb, _stream(stream)), "hca_attend")


def hca_attend_noalloc_scratch_bytes() -> int:
    return int(library().hca_attend_noalloc_scratch_bytes())


def hca_attend_noalloc(q, scale, ck, cv, m, ring_k, ring_v, W, q_pos, out, lse=None, chunk_k=None, chunk_v=None,
                       chunk_pos0=None, splits=0, stream=None):
    """hca_attend for callers that cannot allocate: no workspace argument; the split partials
    live in the library's fixed device scratch (see include/csa_hca.h).  Calls that may
    overlap on the GPU share that scratch and must be serialised by the caller."""
    B, T, H, d = q.shape
    ring_cap = ring_k.shape[1] if ring_k is not None else 0
    ck_, cv_, cp_, cs_ = _chunk_args(chunk_k, chunk_v, chunk_pos0)
    _check(library().hca_attend_noalloc(_p(q), B, T, H, d, float(scale), _p(ck), _p(cv), ck.shape[1], int(m),
                                        _p(ring_k), _p(ring_v), ring_cap, int(W), _p(ck_), _p(cv_), _p(cp_), cs_,
                                        _p(q_pos), int(splits), _kv_dt(q, ck), _p(out), _p(lse), _stream(stream)),
           "hca_attend_noalloc")


def csa_cache_append(k_new, v_new, gate_new, kidx_new, pos, slot_bias, m, ring_k, ring_v, ring_gate, ck, cv,
                     k_codes, k_scale, key_fmt, stream=None):
    """k_new/v_new [B, n_new, d]; gate_new [B, n_new]; kidx_new [B, n_new//m + 1, d_I]; pos int64 [B]."""
    B, n_new, d = k_new.shape
    d_I = kidx_new.shape[-1]
    assert kidx_new.shape[1] == n_new // m + 1
    _check(library().csa_cache_append(_p(k_new), _p(v_new), _p(gate_new), _p(kidx_new), _dt(kidx_new), _p(pos), B, n_new,
                                 d, _kv_dt(k_new, ck), _p(slot_bias), int(m), _p(ring_k), _p(ring_v), _p(ring_gate),
                                 ring_k.shape[1], _p(ck), _p(cv), ck.shape[1], _p(k_codes), _p(k_scale),
                                 int(key_fmt), d_I, _stream(stream)), "csa_cache_append")


def hca_cache_append(k_new, v_new, gate_new, pos, slot_bias, m, ring_k, ring_v, ring_gate, ck, cv, stream=None):
    B, n_new, d = k_new.shape
    _check(library().hca_cache_append(_p(k_new), _p(v_new), _p(gate_new), _p(pos), B, n_new, d, _kv_dt(k_new, ck),
                                 _p(slot_bias), int(m), _p(ring_k), _p(ring_v), _p(ring_gate), ring_k.shape[1],
                                 _p(ck), _p(cv), ck.shape[1], _stream(stream)), "hca_cache_append")


def swa_ring_write(k_new, v_new, gate_new, pos, n_new, ring_k, ring_v, ring_gate, stream=None):
    """k_new/v_new [B, new_stride, d] (first n_new rows used); gate_new [B, new_stride]; pos int64 [B]."""
    B, stride, d = k_new.shape
    _check(library().swa_ring_write(_p(k_new), _p(v_new), _p(gate_new), stride, _p(pos), B, int(n_new), d, _dt(k_new),
                               _p(ring_k), _p(ring_v), _p(ring_gate), ring_k.shape[1], _stream(stream)),
           "swa_ring_write")
