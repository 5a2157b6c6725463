"""Pins for the oracle's index-key quantisation (FP8 e4m3 + row scale; FP4 e2m1 + UE8M0/32).

Low-precision lightning-indexer keys: pogovet.com DeepSeek-V4 article, details 4 and 5
("FP4 기반 lightning indexer"); honbul.tistory.com/221 FP4 QAT section (CSA indexer
query-key path).  Formats: OCP OFP8 v1.0 (E4M3) and OCP MX v1.0 (E2M1, E8M0 scale).
"""
import numpy as np
import pytest
import torch

import oracle
from tests.golden import load


def test_e4m3_code_table_matches_spec_and_library():
    g = load("e4m3_ocp_fp8.txt")
    for c, v in zip(g["codes"], g["values"]):
        got = oracle.e4m3_decode(int(c))
        assert got == v and np.signbit(got) == np.signbit(v)
    for c in g["nan_codes"]:
        assert np.isnan(oracle.e4m3_decode(int(c)))
    # all 256 codes against torch's float8_e4m3fn (independent library decoder)
    codes = torch.arange(256, dtype=torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_decode(c) for c in range(256)])
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(lib))
    ok = ~np.isnan(lib)
    np.testing.assert_array_equal(mine[ok], lib[ok])


def test_e4m3_encode_round_trip_and_rne():
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if np.isnan(v):
            continue
        assert oracle.e4m3_encode(v) == c
    rng = np.random.default_rng(0)
    vals = rng.standard_normal(20000) * 2.0 ** rng.integers(-12, 9, 20000)
    vals = vals[np.abs(vals) < 448.0]
    # midpoints between neighbouring codes must go to the even code
    pos = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    mids = (pos[:-1] + pos[1:]) / 2
    vals = np.concatenate([vals, mids, -mids])
    mine = np.array([oracle.e4m3_encode(v) for v in vals], dtype=np.uint8)
    lib = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(mine, lib)
    for mcode, mid in zip(range(0x7E), mids):
        assert oracle.e4m3_encode(mid) % 2 == 0 and oracle.e4m3_encode(mid) in (mcode, mcode + 1)


def test_e4m3_saturates():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(470.0) == 0x7E
    assert oracle.e4m3_encode(1e9) == 0x7E
    assert oracle.e4m3_encode(-1e9) == 0xFE


def test_e2m1_table_rne_and_saturation():
    g = load("e2m1_ocp_mx.txt")
    for c, v in zip(g["codes"], g["values"]):
        got = oracle.e2m1_decode(int(c))
        assert got == v and np.signbit(got) == np.signbit(v)
        assert oracle.e2m1_encode(v) == int(c)
    for x, y in zip(g["rne_in"], g["rne_out"]):
        got = oracle.e2m1_decode(oracle.e2m1_encode(x))
        assert got == y, (x, got, y)


def test_e4m3_rowscale_quantisation_bounds():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((64, 64)) * 0.125).astype(np.float32)
    x[3] = 0.0                                        # all-zero row -> scale 1, codes 0
    x[5, 7] = 4.0                                     # an outlier
    codes, s = oracle.quant_e4m3_rowscale(x)
    assert s[3] == 1.0 and (codes[3] == 0).all()
    amax = np.abs(x).max(1)
    nz = amax > 0
    np.testing.assert_array_equal(s[nz], (amax[nz] / np.float32(448.0)).astype(np.float32))
    khat = oracle.dequant_keys(oracle.KEY_E4M3, codes, s, 64)
    # |khat - x| <= s * half-ulp: relative 2^-4 for normals, absolute 2^-10 * s for subnormals
    err = np.abs(khat - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, s[:, None].astype(np.float64) * 2.0 ** -10) * (1 + 1e-6)
    assert (err <= bound).all()
    # the largest element of every row lands on the top code 448
    top = np.abs(oracle.dequant_keys(oracle.KEY_E4M3, codes, np.ones_like(s), 64)).max(1)
    assert (top[nz] == 448.0).all()


def test_e2m1_ue8m0_quantisation_bounds_and_idempotence():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((50, 64)).astype(np.float32)
    x[0, :32] = 0.0                                   # zero block -> exponent 0
    x[1, 40] = 37.0                                   # outlier in the second block
    xb = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    packed, se = oracle.quant_e2m1_ue8m0(xb)
    xv = oracle.bf16_to_f64(xb)
    e = se.astype(np.int64) - 127
    amax = np.abs(xv.reshape(50, 2, 32)).max(-1)
    assert e[0, 0] == 0
    nz = amax > 0
    # minimal power of two: amax <= 6*2^e and amax > 6*2^(e-1)
    assert (amax[nz] <= 6.0 * 2.0 ** e[nz]).all() and (amax[nz] > 3.0 * 2.0 ** e[nz]).all()
    khat = oracle.dequant_keys(oracle.KEY_E2M1, packed, se, 64)
    # error <= half the grid spacing at that magnitude (spacing 0.5/1/2 * 2^e)
    sc = np.repeat(2.0 ** e, 32, axis=1)
    y = np.abs(xv) / sc
    half = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0)) * sc
    assert (np.abs(khat - xv) <= half * (1 + 1e-12)).all()
    # packing: the even element sits in the low nibble
    lo = oracle.e2m1_decode(int(packed[1, 0] & 0xF)) * 2.0 ** e[1, 0]
    assert lo == khat[1, 0]
    # quantising the dequantised keys again reproduces the same key values
    p2, s2 = oracle.quant_e2m1_ue8m0(khat.astype(np.float32))
    np.testing.assert_array_equal(oracle.dequant_keys(oracle.KEY_E2M1, p2, s2, 64), khat)


@pytest.mark.parametrize("fmt", [oracle.KEY_F32, oracle.KEY_BF16])
def test_plain_key_formats_pass_through(fmt):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((7, 32)).astype(np.float32)
    if fmt == oracle.KEY_BF16:
        x = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    codes, sc = oracle.quantize_keys(x, fmt)
    np.testing.assert_array_equal(oracle.dequant_keys(fmt, codes, sc, 32), oracle.to_f64(x))
