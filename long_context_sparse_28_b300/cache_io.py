"""On-disk prefix caches: save the state of a CSA or HCA layer cache after a prefix and restore it
into a sequence slot of a cache, so that a request sharing that prefix continues decoding from it
instead of prefilling again (honbul.tistory.com/221, "KV cache를 줄이는 방식": the compressed
cache of a shared prefix is kept on disk and reused, e.g. for many questions on one long document).

The state of sequence b after n_ctx tokens (positions 0 .. n_ctx-1) is, in the split layout of
``layers.py``: the n_ctx // m compressed entries (ck, cv and, for CSA, the index-key codes and
scales) and the whole window ring (ring_k, ring_v, ring_gate; it also holds the tail of the block
being filled).  Nothing else is needed to append token n_ctx and attend from it.  A state must be
saved when the sequence has consumed exactly n_ctx tokens: the ring of a sequence that went on
holds later tokens.

File layout (little-endian): 8-byte magic ``CSAHCAKV``, uint32 format version, uint32 header
length, the header as UTF-8 JSON (geometry, per saved sequence its n_ctx and entry count, and
per stored tensor its name, sequence, dtype, shape, byte offset and size), then the tensors' raw
bytes, each at a 256-byte aligned offset.  Only visible entries are stored; on restore the slot's
entries from n_ctx // m on are zeroed.  Loading checks the magic, version, geometry and every
tensor's bounds, and raises ValueError on any mismatch.  Copies between device and host go
through torch (plain tensor copies); no kernel computes on the state.
"""
from __future__ import annotations

import json
import os
import struct

import numpy as np
import torch

from .layers import CSACache, HCACache

MAGIC = b"CSAHCAKV"
VERSION = 1
_ALIGN = 256
_DTYPES = {"bfloat16": torch.bfloat16, "float32": torch.float32, "uint8": torch.uint8}
_NAMES = {v: k for k, v in _DTYPES.items()}


def _kind(cache) -> str:
    if isinstance(cache, CSACache):
        return "csa"
    if isinstance(cache, HCACache):
        return "hca"
    raise TypeError("expected a CSACache or an HCACache")


def _geometry(cache) -> dict:
    g = {"kind": _kind(cache), "m": int(cache.m), "d": int(cache.d), "W": int(cache.W),
         "dtype": _NAMES[cache.dtype]}
    if g["kind"] == "csa":
        g.update(d_I=int(cache.d_I), key_fmt=int(cache.key_fmt))
    if getattr(cache, "kv_fp8", False):       # compressed K/V rows in FP8 (recorded only when set)
        g["kv_fp8"] = True
    return g


def _seq_tensors(cache, b: int, n_entries: int):
    """(name, tensor view) of sequence b's state: visible entries and the whole ring."""
    out = [("ck", cache.ck[b, :n_entries]), ("cv", cache.cv[b, :n_entries]), ("ring_k", cache.ring_k[b]),
           ("ring_v", cache.ring_v[b]), ("ring_gate", cache.ring_gate[b])]
    if _kind(cache) == "csa":
        out.append(("k_codes", cache.k_codes[b, :n_entries]))
        if cache.k_scale is not None:
            out.append(("k_scale", cache.k_scale[b, :n_entries]))
    return out


def _raw_bytes(t: torch.Tensor) -> bytes:
    t = t.detach().contiguous().cpu()
    return t.view(torch.uint8).numpy().tobytes() if t.numel() else b""


def save_prefix(path: str, cache, n_ctx, seqs=None) -> None:
    """Writes the state of sequences `seqs` (default: all) of `cache` after n_ctx[b] tokens."""
    seqs = list(range(cache.B)) if seqs is None else [int(b) for b in seqs]
    n_ctx = [int(x) for x in (n_ctx if hasattr(n_ctx, "__len__") else [n_ctx] * cache.B)]
    header = dict(_geometry(cache), seqs=[], tensors=[])
    blobs, off = [], 0
    for i, b in enumerate(seqs):
        if not 0 <= b < cache.B:
            raise ValueError(f"sequence {b} outside the cache's {cache.B}")
        n = n_ctx[b]
        ne = n // cache.m
        if n < 0 or ne > cache.Ncap:
            raise ValueError(f"sequence {b}: {n} tokens do not fit the cache ({cache.Ncap} entries)")
        header["seqs"].append({"n_ctx": n, "n_entries": ne})
        for name, t in _seq_tensors(cache, b, ne):
            data = _raw_bytes(t)
            header["tensors"].append({"name": name, "seq": i, "dtype": _NAMES[t.dtype], "shape": list(t.shape),
                                      "offset": off, "nbytes": len(data)})
            blobs.append((off, data))
            off += (len(data) + _ALIGN - 1) // _ALIGN * _ALIGN
    hdr = json.dumps(header).encode()
    start = (16 + len(hdr) + _ALIGN - 1) // _ALIGN * _ALIGN
    tmp = path + ".tmp"
    with open(tmp, "wb") as f:
        f.write(MAGIC + struct.pack("<II", VERSION, len(hdr)) + hdr)
        end = start
        for o, data in blobs:
            f.seek(start + o)
            f.write(data)
            end = max(end, start + o + len(data))
        f.truncate(end)
    os.replace(tmp, path)


def read_header(path: str) -> tuple[dict, int]:
    """The file's header and the byte offset of its tensor data; ValueError if it is not a
    prefix-cache file of this version."""
    with open(path, "rb") as f:
        head = f.read(16)
        if len(head) < 16 or head[:8] != MAGIC:
            raise ValueError(f"{path}: not a prefix-cache file")
        version, n = struct.unpack("<II", head[8:])
        if version != VERSION:
            raise ValueError(f"{path}: format version {version}, expected {VERSION}")
        raw = f.read(n)
    if len(raw) != n:
        raise ValueError(f"{path}: truncated header")
    try:
        header = json.loads(raw.decode())
    except (UnicodeDecodeError, json.JSONDecodeError) as e:
        raise ValueError(f"{path}: unreadable header ({e})") from None
    _check_schema(path, header)
    return header, (16 + n + _ALIGN - 1) // _ALIGN * _ALIGN


def _is_int(x) -> bool:
    return isinstance(x, int) and not isinstance(x, bool)


def _check_schema(path: str, h) -> None:
    """Every field the loaders use is present, of the right type and in range."""
    def bad(what):
        raise ValueError(f"{path}: malformed header ({what})")
    if not isinstance(h, dict):
        bad("not an object")
    if h.get("kind") not in ("csa", "hca"):
        bad("kind")
    if h.get("dtype") not in _DTYPES:
        bad("dtype")
    if "kv_fp8" in h and not isinstance(h["kv_fp8"], bool):
        bad("kv_fp8")
    for key in ("m", "d", "W") + (("d_I", "key_fmt") if h["kind"] == "csa" else ()):
        if not _is_int(h.get(key)) or h[key] < 0:
            bad(key)
    seqs, tensors = h.get("seqs"), h.get("tensors")
    if not isinstance(seqs, list) or not isinstance(tensors, list):
        bad("seqs / tensors")
    for sq in seqs:
        if not isinstance(sq, dict) or not _is_int(sq.get("n_ctx")) or not _is_int(sq.get("n_entries")) \
                or sq["n_ctx"] < 0 or sq["n_entries"] < 0:
            bad("sequence entry")
    for e in tensors:
        if not isinstance(e, dict) or not isinstance(e.get("name"), str) or e.get("dtype") not in _DTYPES:
            bad("tensor entry")
        if not _is_int(e.get("seq")) or not 0 <= e["seq"] < len(seqs):
            bad("tensor sequence")
        shape = e.get("shape")
        if not isinstance(shape, list) or not all(_is_int(x) and x >= 0 for x in shape):
            bad("tensor shape")
        if not _is_int(e.get("offset")) or not _is_int(e.get("nbytes")) or e["offset"] < 0 or e["nbytes"] < 0:
            bad("tensor offset / size")


def _load_seq(path, header, start, i):
    """Sequence i's tensors from the file as CPU tensors, checked against the header."""
    size = os.path.getsize(path)
    out = {}
    with open(path, "rb") as f:
        for e in header["tensors"]:
            if e["seq"] != i:
                continue
            dt = _DTYPES.get(e["dtype"])
            if dt is None:
                raise ValueError(f"{path}: unknown dtype {e['dtype']}")
            shape = [int(s) for s in e["shape"]]
            nbytes = int(np.prod(shape)) * torch.empty(0, dtype=dt).element_size()
            if nbytes != e["nbytes"] or e["offset"] < 0 or start + e["offset"] + nbytes > size:
                raise ValueError(f"{path}: tensor {e['name']} of sequence {i} is out of bounds or inconsistent")
            f.seek(start + e["offset"])
            data = f.read(nbytes)
            t = torch.frombuffer(bytearray(data), dtype=torch.uint8) if nbytes else torch.empty(0, dtype=torch.uint8)
            out[e["name"]] = t.view(dt).reshape(shape)
    return out


def load_prefix_into(path: str, cache, b: int, seq: int = 0) -> int:
    """Restores saved sequence `seq` of the file into slot b of `cache` (same geometry; the
    cache's capacity may differ) and returns its n_ctx: the slot's next token is at position
    n_ctx.  Entries of the slot from n_ctx // m on are zeroed."""
    header, start = read_header(path)
    g = _geometry(cache)
    for key, val in g.items():
        if header.get(key) != val:
            raise ValueError(f"{path}: {key} = {header.get(key)!r}, the cache has {val!r}")
    if bool(header.get("kv_fp8", False)) != bool(g.get("kv_fp8", False)):
        raise ValueError(f"{path}: kv_fp8 = {header.get('kv_fp8', False)!r}, the cache has {g.get('kv_fp8', False)!r}")
    if not 0 <= seq < len(header["seqs"]):
        raise ValueError(f"{path}: no saved sequence {seq}")
    if not 0 <= b < cache.B:
        raise ValueError(f"slot {b} outside the cache's {cache.B}")
    s = header["seqs"][seq]
    n_ctx, ne = int(s["n_ctx"]), int(s["n_entries"])
    if n_ctx < 0 or ne != n_ctx // cache.m or ne > cache.Ncap:
        raise ValueError(f"{path}: sequence {seq} ({n_ctx} tokens, {ne} entries) does not fit the cache")
    data = _load_seq(path, header, start, seq)
    want = {name: tuple(t.shape) for name, t in _seq_tensors(cache, b, ne)}
    got = {name: tuple(t.shape) for name, t in data.items()}
    if want != got:
        raise ValueError(f"{path}: stored tensors {got} do not match the cache's {want}")
    for name, dst in _seq_tensors(cache, b, ne):
        dst.copy_(data[name])
    cache.ck[b, ne:].zero_()
    cache.cv[b, ne:].zero_()
    if g["kind"] == "csa":
        cache.k_codes[b, ne:].zero_()
        if cache.k_scale is not None:
            cache.k_scale[b, ne:].zero_()
    return n_ctx


def load_prefix(path: str, device="cuda", Ncap: int | None = None):
    """A new cache holding every sequence saved in the file (capacity Ncap, default: the
    largest saved entry count) and the list of their n_ctx."""
    header, _ = read_header(path)
    ns = [int(s["n_entries"]) for s in header["seqs"]]
    Ncap = max(ns + [1]) if Ncap is None else int(Ncap)
    dt = _DTYPES[header["dtype"]]
    B = len(ns)
    fp8 = bool(header.get("kv_fp8", False))
    if header["kind"] == "csa":
        cache = CSACache(B, Ncap, header["d"], header["W"], header["d_I"], header["key_fmt"], dt, device,
                         m=header["m"], kv_fp8=fp8)
    elif header["kind"] == "hca":
        cache = HCACache(B, Ncap, header["d"], header["W"], dt, device, m=header["m"], kv_fp8=fp8)
    else:
        raise ValueError(f"{path}: unknown cache kind {header['kind']!r}")
    return cache, [load_prefix_into(path, cache, i, i) for i in range(B)]
