"""CPU checks of the C-ABI boundary: the library loads, exports every declared entry point,
and rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


def _declared():
    names = []
    pat = re.compile(r"^\s*(?:csahca_status|size_t|const char\s*\*|uint64_t|int)\s+(\w+)\s*\(", re.M)
    for h in HEADERS:
        names += pat.findall(open(h).read())
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from long_context_sparse_28_b300 import build_lib
    path = build_lib.build()
    return ctypes.CDLL(path)


def test_header_declares_the_method_entry_points():
    names = _declared()
    for n in ["csa_compress", "hca_compress", "csa_index_topk", "csa_attend", "hca_attend", "csa_cache_append",
              "hca_cache_append", "csa_index_key_quantize", "csa_topk_from_scores", "csahca_device_status"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_binding_exposes_every_symbol():
    import long_context_sparse_28_b300 as m
    for n in _declared():
        if n.startswith("csahca_"):
            continue
        assert callable(getattr(m, n)), n


def test_host_validation_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    lib.csa_compress.argtypes = [P, P, P, ctypes.c_int64, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int, P, P, ctypes.c_int64, P]
    # null pointers -> CSAHCA_ERR_INVALID_ARG (1), nothing launched
    assert lib.csa_compress(None, None, None, 16, None, None, None, 4, 1, 128, 1, None, None, 4, None) == 1
    lib.csa_topk_from_scores.argtypes = [P, ctypes.c_int64, ctypes.c_int, P, ctypes.c_int, P, P, ctypes.c_size_t, P]
    fake = ctypes.c_void_p(256)
    # k = 0 is invalid
    assert lib.csa_topk_from_scores(fake, 10, 1, fake, 0, fake, fake, 1 << 20, None) == 1
    # workspace too small -> CSAHCA_ERR_WORKSPACE (6)
    assert lib.csa_topk_from_scores(fake, 10, 1, fake, 4, fake, fake, 16, None) == 6
    lib.csahca_status_string.restype = ctypes.c_char_p
    assert lib.csahca_status_string(6) == b"workspace missing, too small or misaligned"


def test_workspace_sizes_are_host_only(lib):
    lib.csa_index_topk_workspace.restype = ctypes.c_size_t
    lib.csa_index_topk_workspace.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int]
    n = lib.csa_index_topk_workspace(32, 1, 262144, 1024)
    # scores (32 x 262144 fp32) + the 12-bit histograms + 2 bitmaps per row
    assert n >= 32 * 262144 * 4 + 32 * 4096 * 4 + 2 * 32 * 8192 * 4
    lib.hca_attend_workspace.restype = ctypes.c_size_t
    lib.hca_attend_workspace.argtypes = [ctypes.c_int] * 4 + [ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    # per-row arrival counters (65536 x 4 B) + partial outputs + partial log-sum-exps
    assert lib.hca_attend_workspace(4, 1, 64, 128, 8192, 128, 8) == 65536 * 4 + 4 * 8 * 64 * 128 * 4 + 4 * 8 * 64 * 4
