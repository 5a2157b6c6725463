"""On-disk prefix caches (CPU): a saved layer-cache state restores bit for bit, into a new cache
or into one slot of an existing cache, and damaged or mismatched files are refused."""
import struct

import pytest
import torch

import long_context_sparse_28_b300 as L
from long_context_sparse_28_b300 import cache_io
from long_context_sparse_28_b300.layers import CSACache, HCACache


def _fill(cache, seed):
    g = torch.Generator().manual_seed(seed)
    for name in ("ck", "cv", "ring_k", "ring_v", "ring_gate", "k_codes", "k_scale"):
        t = getattr(cache, name, None)
        if t is None:
            continue
        if t.dtype == torch.uint8:
            t.copy_(torch.randint(0, 256, t.shape, generator=g, dtype=torch.uint8))
        else:
            t.copy_(torch.randn(t.shape, generator=g).to(t.dtype))
    return cache


def _state(cache, b, n_ctx):
    ne = n_ctx // cache.m
    return {k: v.clone() for k, v in cache_io._seq_tensors(cache, b, ne)}


def _same(a, b):
    assert a.keys() == b.keys()
    for k in a:
        assert a[k].dtype == b[k].dtype and a[k].shape == b[k].shape, k
        assert torch.equal(a[k].contiguous().view(torch.uint8), b[k].contiguous().view(torch.uint8)), k


@pytest.mark.parametrize("fmt", ["e2m1", "e4m3", "bf16"])
def test_csa_prefix_round_trip(tmp_path, fmt):
    src = _fill(CSACache(3, 40, 64, 16, 64, L.KEY_FMT[fmt], torch.bfloat16, "cpu"), 1)
    n_ctx = [130, 3, 0]                                       # 32 entries; window only; empty
    p = str(tmp_path / "csa.kv")
    cache_io.save_prefix(p, src, n_ctx)
    dst, got = cache_io.load_prefix(p, device="cpu")
    assert got == n_ctx
    for b in range(3):
        _same(_state(src, b, n_ctx[b]), _state(dst, b, n_ctx[b]))
        ne = n_ctx[b] // src.m
        assert not dst.ck[b, ne:].any() and not dst.k_codes[b, ne:].any()


def test_hca_prefix_into_a_slot_of_a_running_cache(tmp_path):
    src = _fill(HCACache(2, 9, 32, 128, torch.float32, "cpu"), 2)
    p = str(tmp_path / "hca.kv")
    cache_io.save_prefix(p, src, [128 * 7 + 5, 50], seqs=[0])
    dst = _fill(HCACache(4, 12, 32, 128, torch.float32, "cpu"), 3)   # larger capacity, other contents
    before = _state(dst, 3, 128 * 12)
    n = cache_io.load_prefix_into(p, dst, 1, seq=0)
    assert n == 128 * 7 + 5
    _same(_state(src, 0, n), _state(dst, 1, n))
    assert not dst.ck[1, 7:].any() and not dst.cv[1, 7:].any()       # stale entries cleared
    _same(before, _state(dst, 3, 128 * 12))                           # other slots untouched


def test_damaged_or_mismatched_files_are_refused(tmp_path):
    # CSA caches hold whole 256-entry stages: capacity 512 here, 256 for the small one below
    src = _fill(CSACache(1, 300, 64, 16, 64, L.KEY_FMT["e2m1"], torch.bfloat16, "cpu"), 4)
    p = tmp_path / "a.kv"
    cache_io.save_prefix(str(p), src, [4 * 300])
    raw = p.read_bytes()
    bad = tmp_path / "bad.kv"
    bad.write_bytes(b"XXXXXXXX" + raw[8:])
    with pytest.raises(ValueError, match="not a prefix-cache file"):
        cache_io.load_prefix(str(bad), device="cpu")
    bad.write_bytes(raw[:8] + struct.pack("<I", 99) + raw[12:])
    with pytest.raises(ValueError, match="version"):
        cache_io.load_prefix(str(bad), device="cpu")
    bad.write_bytes(raw[: len(raw) - 100])
    with pytest.raises(ValueError, match="out of bounds"):
        cache_io.load_prefix(str(bad), device="cpu")
    other = CSACache(1, 300, 64, 16, 64, L.KEY_FMT["e4m3"], torch.bfloat16, "cpu")
    with pytest.raises(ValueError, match="key_fmt"):
        cache_io.load_prefix_into(str(p), other, 0)
    small = CSACache(1, 8, 64, 16, 64, L.KEY_FMT["e2m1"], torch.bfloat16, "cpu")
    with pytest.raises(ValueError, match="does not fit"):
        cache_io.load_prefix_into(str(p), small, 0)
    with pytest.raises(ValueError, match="do not fit"):
        cache_io.save_prefix(str(tmp_path / "c.kv"), src, [4 * 513])


def _rewrite_header(raw: bytes, header: dict) -> bytes:
    """The file with its JSON header replaced (tensor data re-aligned after it)."""
    import json
    n = struct.unpack("<I", raw[12:16])[0]
    start = (16 + n + 255) // 256 * 256
    hdr = json.dumps(header).encode()
    new_start = (16 + len(hdr) + 255) // 256 * 256
    return raw[:12] + struct.pack("<I", len(hdr)) + hdr + b"\0" * (new_start - 16 - len(hdr)) + raw[start:]


@pytest.mark.parametrize("edit", ["drop_seqs", "drop_dtype", "bad_kind", "tensor_no_seq", "negative_shape",
                                  "seq_out_of_range", "shape_not_list", "not_object"])
def test_malformed_headers_are_refused_with_value_error(tmp_path, edit):
    src = _fill(HCACache(2, 8, 64, 16, torch.bfloat16, "cpu", m=128), 6)
    p = tmp_path / "a.kv"
    cache_io.save_prefix(str(p), src, [128 * 3, 128 * 2])
    raw = p.read_bytes()
    header, _ = cache_io.read_header(str(p))
    h = dict(header)
    t0 = dict(h["tensors"][0])
    if edit == "drop_seqs":
        del h["seqs"]
    elif edit == "drop_dtype":
        del h["dtype"]
    elif edit == "bad_kind":
        h["kind"] = "mla"
    elif edit == "tensor_no_seq":
        del t0["seq"]
    elif edit == "negative_shape":
        t0["shape"] = [-3, 64]
    elif edit == "seq_out_of_range":
        t0["seq"] = 5
    elif edit == "shape_not_list":
        t0["shape"] = "3x64"
    h["tensors"] = [t0] + h["tensors"][1:]
    if edit == "not_object":
        h = [1, 2, 3]
    bad = tmp_path / "bad.kv"
    bad.write_bytes(_rewrite_header(raw, h))
    with pytest.raises(ValueError):
        cache_io.load_prefix(str(bad), device="cpu")
    dst = HCACache(2, 8, 64, 16, torch.bfloat16, "cpu", m=128)
    with pytest.raises(ValueError):
        cache_io.load_prefix_into(str(bad), dst, 0)


def test_fp8_cache_round_trip_and_mismatch(tmp_path):
    # FP8 compressed K/V rows (uint8) are saved and restored as bytes; the flag travels in the
    # header, and a bf16 cache refuses an FP8 file
    src = _fill(CSACache(2, 40, 128, 16, 64, L.KEY_FMT["e2m1"], torch.bfloat16, "cpu", kv_fp8=True), 7)
    assert src.ck.dtype == torch.uint8 and src.ck.shape[-1] == L.KV_FP8_K_ROW
    p = str(tmp_path / "fp8.kv")
    cache_io.save_prefix(p, src, [4 * 33 + 1, 9])
    dst, got = cache_io.load_prefix(p, device="cpu")
    assert dst.kv_fp8 and got == [4 * 33 + 1, 9]
    for b, n in enumerate(got):
        _same(_state(src, b, n), _state(dst, b, n))
    plain = CSACache(2, 40, 128, 16, 64, L.KEY_FMT["e2m1"], torch.bfloat16, "cpu")
    with pytest.raises(ValueError, match="kv_fp8"):
        cache_io.load_prefix_into(p, plain, 0)
    p2 = str(tmp_path / "bf16.kv")
    cache_io.save_prefix(p2, _fill(plain, 8), [4 * 20, 0])
    with pytest.raises(ValueError, match="kv_fp8"):
        cache_io.load_prefix_into(p2, src, 0)


def test_fp8_hca_prefix_into_a_slot(tmp_path):
    src = _fill(HCACache(2, 9, 128, 128, torch.bfloat16, "cpu", kv_fp8=True), 8)
    p = str(tmp_path / "hca8.kv")
    cache_io.save_prefix(p, src, [128 * 6 + 3, 128])
    dst = _fill(HCACache(3, 12, 128, 128, torch.bfloat16, "cpu", kv_fp8=True), 9)
    n = cache_io.load_prefix_into(p, dst, 2, seq=0)
    assert n == 128 * 6 + 3
    _same(_state(src, 0, n), _state(dst, 2, n))
    assert not dst.ck[2, 6:].any() and not dst.cv[2, 6:].any()
